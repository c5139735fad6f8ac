// One-shot KV compaction for sm_103a (FastKV, 2.B Decoupled KV Retention): destination row r of
// (layer, b, h) receives source row idx_layer[b, h, r] for r < k (one set shared by all layers, or one
// per layer), then the tail rows tail_lo .. len-1.
//
// Pure data movement: 16 threads move one 256-byte row of K and one of V with 16-byte vector loads
// and stores; each thread handles kRowsPerThread rows so several loads are in flight before the
// stores.  Grid: (row blocks, Hkv, B * n_layers).
#include <stdint.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr int kCpThreads = 256;
constexpr int kRowsPerIter = kCpThreads / 16;   // 16 rows per CTA pass
constexpr int kRowsPerThread = 4;

__device__ __forceinline__ uint4 ld_nc16(const uint16_t* ptr)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(ptr));
    return r;
}

__global__ void __launch_bounds__(kCpThreads) compact_kernel(const CompactParams p)
{
    griddep_wait();
    griddep_launch();
    const int h = blockIdx.y;
    const int b = blockIdx.z % p.B;
    const int layer = blockIdx.z / p.B;
    const int sub = threadIdx.x & 15;
    const int rloc = threadIdx.x >> 4;

    int lenb = p.len[b];
    if (lenb < 0 || lenb > p.Tcap) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0 && layer == 0) atomicOr(p.err, FX_DEVERR_LEN);
        lenb = lenb < 0 ? 0 : p.Tcap;
    }
    int nrows = p.kk + max(0, lenb - p.tail_lo);
    if (blockIdx.x == 0 && h == 0 && layer == 0 && threadIdx.x == 0) {
        if (nrows > p.dcap) atomicOr(p.err, FX_DEVERR_CAPACITY);
        p.dlen[b] = min(nrows, p.dcap);
    }
    nrows = min(nrows, p.dcap);

    const uint16_t* sk = p.sk + layer * p.s_layer + b * p.sb + h * p.sh;
    const uint16_t* sv = p.sv + layer * p.s_layer + b * p.sb + h * p.sh;
    uint16_t* dk = p.dk + layer * p.d_layer + b * p.db + h * p.dh;
    uint16_t* dv = p.dv + layer * p.d_layer + b * p.db + h * p.dh;
    const int32_t* irow = p.idx ? p.idx + layer * p.idx_layer + ((int64_t)b * p.Hkv + h) * p.kk : nullptr;

    const int rbase = blockIdx.x * (kRowsPerIter * kRowsPerThread);
    uint4 kv[kRowsPerThread], vv[kRowsPerThread];
    int dst_row[kRowsPerThread];
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        const int r = rbase + u * kRowsPerIter + rloc;
        dst_row[u] = -1;
        if (r >= nrows) continue;
        int t;
        if (r < p.kk) {
            t = irow[r];
            if (t < 0 || t >= lenb) {
                if (sub == 0) atomicOr(p.err, FX_DEVERR_INDEX);
                continue;
            }
        } else {
            t = p.tail_lo + (r - p.kk);
        }
        kv[u] = ld_nc16(sk + (int64_t)t * p.st + sub * 8);
        vv[u] = ld_nc16(sv + (int64_t)t * p.st + sub * 8);
        dst_row[u] = r;
    }
#pragma unroll
    for (int u = 0; u < kRowsPerThread; ++u) {
        if (dst_row[u] < 0) continue;
        *reinterpret_cast<uint4*>(dk + (int64_t)dst_row[u] * p.dt + sub * 8) = kv[u];
        *reinterpret_cast<uint4*>(dv + (int64_t)dst_row[u] * p.dt + sub * 8) = vv[u];
    }
}

// Decode-step append: one warp per (layer, b, h) row pair; lanes 0..15 copy the 16-byte chunks of the
// new K row, lanes 16..31 those of the V row, into row pos[b] of that layer's cache.
__global__ void __launch_bounds__(kCpThreads) append_kernel(const AppendParams p)
{
    griddep_wait();   // the new rows may come from the kernel just before
    griddep_launch();
    const int64_t w = (int64_t)blockIdx.x * (kCpThreads / 32) + (threadIdx.x >> 5);
    const int64_t rows = (int64_t)p.n_layers * p.B * p.Hkv;
    if (w >= rows) return;
    const int lane = threadIdx.x & 31;
    const int h = (int)(w % p.Hkv);
    const int64_t lb = w / p.Hkv;
    const int b = (int)(lb % p.B);
    const int l = (int)(lb / p.B);
    const int t = p.pos[b];
    if (t < 0 || t >= p.Tcap) {
        if (lane == 0 && h == 0 && l == 0) atomicOr(p.err, FX_DEVERR_LEN);
        return;
    }
    const int c = lane & 15;
    const uint16_t* src = (lane < 16 ? p.k_new : p.v_new) + (w << 7) + 8 * c;
    uint16_t* dst = (lane < 16 ? p.k : p.v) + l * p.layer + b * p.sb + h * p.sh + (int64_t)t * p.st + 8 * c;
    *reinterpret_cast<uint4*>(dst) = ld_nc16(src);
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, bool pdl, cudaStream_t s)
{
    const int64_t rows = (int64_t)p.n_layers * p.B * p.Hkv;
    const int per_cta = kCpThreads / 32;
    dim3 grid((unsigned)((rows + per_cta - 1) / per_cta));
    return launch_kernel(append_kernel, grid, dim3(kCpThreads), 0, s, pdl, 0u, p);
}

cudaError_t launch_compact(const CompactParams& p, bool pdl, cudaStream_t s)
{
    const int rows_per_cta = kRowsPerIter * kRowsPerThread;
    dim3 grid((p.max_rows + rows_per_cta - 1) / rows_per_cta, p.Hkv, p.B * p.n_layers);
    if (grid.x == 0) grid.x = 1;
    return launch_kernel(compact_kernel, grid, dim3(kCpThreads), 0, s, pdl, 0u, p);
}

}  // namespace fx
