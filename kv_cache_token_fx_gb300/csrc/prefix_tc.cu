// Dense shared-prefix attention on the tensor cores of sm_103a (tcgen05, accumulators in tensor memory).
//
// HPD-Parsing (part 2, shared-prefix KV reuse; part 3, parallel verification of drafted tokens): every
// branch attends over the same prefix rows (up to its fork position) before its own suffix and drafts.
// Per KV head the query rows of all branches (Br x R of them) therefore meet one shared set of keys --
// a real matrix product, which this kernel runs as 128 x 128 tiles on the tensor cores:
//   S = Q K^T       (M = 128 query rows, N = 128 prefix keys, K = 128 dims)        -> tensor memory
//   O += P V        (M = 128 query rows, N = 128 dims, K = 128 prefix keys)        -> tensor memory
// in one pass with an online softmax (P = exp2(S - m) against a running maximum m that moves only by
// more than a fixed slack, so O is rescaled rarely), P split into bf16 hi + lo parts (two products) so
// the probabilities keep about 16 bits.  Two threads own one query row, each for half of
// the keys of a tile and half of O: they read their S columns from tensor memory, trade the row
// maximum, form P, and write it to shared memory as the next product's A operand.  Operand tiles are
// K-major with the 128-byte swizzle; V is transposed into that layout through ldmatrix / stmatrix.trans.
// The result per row is a partial (m, l, O) over the prefix, which the verify kernel folds into its
// merge of the suffix and draft keys.
#include <cuda_bf16.h>
#include <stdint.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr int kTcRows = 128;                       // query rows per CTA (one tensor-memory lane each)
constexpr int kTcKeys = 128;                       // prefix keys per tile
constexpr int kTcThreads = 256;                   // two threads per query row
constexpr int kTileBytes = kTcRows * kHeadDim * 2;  // one 128 x 128 bf16 operand tile
constexpr int kVsPitch = 272;                      // V staging row pitch: conflict-free ldmatrix
constexpr int kTmemCols = 256;                     // S in columns 0..127, O in 128..255
// [Q | K | V^T | P_hi | P_lo] swizzled tiles, the V staging rows, and slack to align to 1024 bytes
constexpr size_t kTcSmem = 5 * (size_t)kTileBytes + (size_t)kTcKeys * kVsPitch + 1024;

// Byte offset of element (r, k) of a [rows x 128] bf16 tile stored K-major with the 128-byte swizzle:
// two 64-wide K blocks of rows x 128 bytes each; 8-row groups of 1024 bytes; within a row the 16-byte
// chunk index is XORed with (row % 8).
__device__ __forceinline__ uint32_t sw128(int r, int k, int rows)
{
    const int kk = k & 63;
    return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((kk >> 3) ^ (r & 7)) << 4) +
                      (kk & 7) * 2);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) (+)= A (smem tile) x B (smem tile)^T over 128 of K, as 8 products of K = 16.
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile, bool accumulate)
{
    constexpr uint32_t idesc = idesc_bf16(128, 128);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (uint32_t)((ks >> 2) * 128 * 128 + (ks & 3) * 32);
        const uint64_t da = sdesc(a_tile + off);
        const uint64_t db = sdesc(b_tile + off);
        const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(da), "l"(db), "r"(idesc), "r"(acc));
    }
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Bounded wait for the products committed to `bar`; flags a timeout instead of hanging.
__device__ __forceinline__ void mma_wait(uint64_t* bar, unsigned& phase, unsigned* err)
{
    unsigned spins = 0, done = 0;
    while (!done) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(phase)
            : "memory");
        if (!done && ++spins == kSpinLimit) {
            if (threadIdx.x == 0) atomicOr(err, FX_DEVERR_TIMEOUT);
            break;
        }
    }
    phase ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, float (&v)[32])
{
    uint32_t u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
          "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]),
          "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
}

// Store 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st32(uint32_t addr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(addr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ float exp2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Everything the products read from shared memory was written by this CTA's threads (generic
// proxy); make it visible to the tensor cores and order it before the one thread that issues them.
__device__ __forceinline__ void publish_to_tensor_core()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1) prefix_tc_kernel(const PrefixTcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char* sQ = base;
    unsigned char* sK = base + kTileBytes;
    unsigned char* sVt = base + 2 * kTileBytes;
    unsigned char* sPh = base + 3 * kTileBytes;
    unsigned char* sPl = base + 4 * kTileBytes;
    unsigned char* sVs = base + 5 * kTileBytes;
    __shared__ __align__(8) uint64_t bar_s;   // S = Q K^T of the current tile is in tensor memory
    __shared__ __align__(8) uint64_t bar_o;   // O += P V of the previous tile is done
    __shared__ uint32_t s_tmem;
    __shared__ int s_lim_max;
    __shared__ float s_xch[kTcThreads];       // the two halves of a row trade their maxima / sums

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int lrow = tid & (kTcRows - 1);     // query row within the tile = tensor-memory lane
    const int half = tid >> 7;                // this thread's 64 keys of each tile and 64 dims of O
    const int col0 = half * 64;
    const int h = blockIdx.y;
    const int rows_total = p.Br * p.R;
    const int row = blockIdx.x * kTcRows + lrow;
    const bool live = row < rows_total;
    const int b = live ? row / p.R : 0;
    const int r = live ? row - b * p.R : 0;

    griddep_wait();   // the queries may come from the kernel just before
    griddep_launch();

    // visible prefix rows of this row's branch (its fork position)
    int lim = 0;
    if (live) {
        lim = p.P;
        if (p.pre_len != nullptr) {
            lim = p.pre_len[b];
            if (lim < 0 || lim > p.P) {
                if (half == 0) atomicOr(p.err, FX_DEVERR_LEN);
                lim = lim < 0 ? 0 : p.P;
            }
        }
    }
    if (tid == 0) {
        s_lim_max = 0;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar_s)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar_o)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // this row's query into the Q tile (zero past the last row); each half copies 64 dims
    {
        const int gi = r / p.Mq;
        const int i = r - gi * p.Mq;
        const uint16_t* qrow = p.q + ((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int d = col0 + 8 * c;
            const uint4 v = live ? *reinterpret_cast<const uint4*>(qrow + d) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sQ + sw128(lrow, d, kTcRows)) = v;
        }
    }
    __syncthreads();
    atomicMax(&s_lim_max, lim);
    publish_to_tensor_core();
    const uint32_t tmem = s_tmem;
    const uint32_t tmem_s = tmem + col0;          // this thread's S columns (S: columns 0..127)
    const uint32_t tmem_o = tmem + 128 + col0;    // this thread's O columns (O: columns 128..255)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int ntiles = (s_lim_max + kTcKeys - 1) / kTcKeys;
    const uint16_t* kb = p.pk + (int64_t)h * p.p_sh;
    const uint16_t* vb = p.pv + (int64_t)h * p.p_sh;

    // K rows into the swizzled K tile, V rows into the staging rows; keys past P are zero
    auto load_k = [&](int j0) {
        for (int e = tid; e < kTcKeys * 16; e += kTcThreads) {
            const int key = e >> 4;
            const int c = e & 15;
            unsigned char* dst = sK + sw128(key, 8 * c, kTcKeys);
            if (j0 + key < p.P)
                cp16(smem_addr(dst), kb + (int64_t)(j0 + key) * p.p_st + 8 * c);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto load_v = [&](int j0) {
        for (int e = tid; e < kTcKeys * 16; e += kTcThreads) {
            const int key = e >> 4;
            const int c = e & 15;
            unsigned char* dst = sVs + key * kVsPitch + 16 * c;
            if (j0 + key < p.P)
                cp16(smem_addr(dst), vb + (int64_t)(j0 + key) * p.p_st + 8 * c);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    // One pass over the prefix with an online softmax.  A row's running maximum m moves only when a
    // tile's maximum exceeds it by more than kMaxSlack (log2 units): O in tensor memory is then rescaled
    // by the row's own threads (read, scale, write back), which happens a few times per row at most, and
    // P = exp2(s - m) stays below 2^kMaxSlack.  The next tile's K and V rows are in flight while this
    // tile's softmax and P V run.
    float m = -INFINITY;
    float l = 0.f;   // this half's share of the row sum
    unsigned ph_s = 0, ph_o = 0;
    if (ntiles > 0) {
        load_k(0);
        load_v(0);
    }
    for (int t = 0; t < ntiles; ++t) {
        const int j0 = t * kTcKeys;
        asm volatile("cp.async.wait_group 1;" ::: "memory");   // K of this tile landed
        publish_to_tensor_core();
        if (tid == 0) {
            mma_tile(tmem, smem_addr(sQ), smem_addr(sK), false);
            mma_commit(&bar_s);
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");   // V of this tile landed
        if (t > 0) mma_wait(&bar_o, ph_o, p.err);               // previous P V done: V^T, P tiles and O free
        __syncthreads();
        // V (keys x dims, staged row-major) -> V^T (dims x keys) in the swizzled K-major layout:
        // 8 x 8 blocks through ldmatrix and stmatrix.trans; warp w owns keys 16w .. 16w+15
        {
            const int j = lane >> 3;
            const int i = lane & 7;
#pragma unroll
            for (int kg = 0; kg < 2; ++kg) {
                const int k0 = warp * 16 + kg * 8;
#pragma unroll
                for (int dq = 0; dq < 4; ++dq) {
                    const int d0 = dq * 32;
                    uint32_t x0, x1, x2, x3;
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                                 : "r"(smem_addr(sVs + (k0 + i) * kVsPitch + (d0 + 8 * j) * 2)));
                    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(
                                     smem_addr(sVt + sw128(d0 + 8 * j + i, k0, kHeadDim))),
                                 "r"(x0), "r"(x1), "r"(x2), "r"(x3)
                                 : "memory");
                }
            }
        }
        mma_wait(&bar_s, ph_s, p.err);   // S of this tile in tensor memory; the K tile is consumed
        __syncthreads();                 // and every warp is done with the V staging rows
        if (t + 1 < ntiles) {
            load_k(j0 + kTcKeys);
            load_v(j0 + kTcKeys);
        }

        // this half's 64 scaled logits, the row's maximum over the tile, and the rescale of O when the
        // running maximum moves
        float sv[2][32];
        tmem_ld32(tmem_s + lane_base, sv[0]);
        tmem_ld32(tmem_s + lane_base + 32, sv[1]);
        const int nv = lim - (j0 + col0);   // keys of this half that the row sees
        float mt = -INFINITY;
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const float x = sv[u][jj] * p.qscale;
                sv[u][jj] = x;
                if (32 * u + jj < nv) mt = fmaxf(mt, x);
            }
        s_xch[tid] = mt;
        __syncthreads();
        mt = fmaxf(mt, s_xch[tid ^ kTcRows]);
        const bool grow = mt > m + kMaxSlack;   // also when m is still -inf and the tile has keys
        const float mnew = grow ? mt : m;
        if (t > 0 && __any_sync(0xffffffffu, grow)) {   // tensor-memory access is warp-wide
            const float a = !grow ? 1.f : (m == -INFINITY ? 0.f : exp2_approx(m - mnew));
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float v[32];
                tmem_ld32(tmem_o + lane_base + 32 * u, v);
#pragma unroll
                for (int c = 0; c < 32; ++c) v[c] *= a;
                tmem_st32(tmem_o + lane_base + 32 * u, v);
            }
            l *= a;
        }
        m = mnew;
        const float ms = (m == -INFINITY) ? 0.f : m;

        // P = exp2(s - m) as bf16 hi + lo into the two P tiles, l += sum P
#pragma unroll
        for (int q = 0; q < 8; ++q) {   // 8 keys = one 16-byte chunk of the P tiles
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float pv[2];
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {
                    const int e = 8 * q + 2 * u + w2;
                    pv[w2] = (e < nv) ? exp2_approx(sv[e >> 5][e & 31] - ms) : 0.f;
                    l += pv[w2];
                }
                __nv_bfloat162 hv = __floats2bfloat162_rn(pv[0], pv[1]);
                hi[u] = *reinterpret_cast<uint32_t*>(&hv);
                lo[u] = pack2_bf16(pv[0] - __low2float(hv), pv[1] - __high2float(hv));
            }
            const uint32_t off = sw128(lrow, col0 + 8 * q, kTcRows);
            *reinterpret_cast<uint4*>(sPh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sPl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        publish_to_tensor_core();   // also: every thread has read S before the next tile overwrites it
        if (tid == 0) {
            mma_tile(tmem + 128, smem_addr(sPh), smem_addr(sVt), t > 0);
            mma_tile(tmem + 128, smem_addr(sPl), smem_addr(sVt), true);
            mma_commit(&bar_o);
        }
    }
    if (ntiles > 0) mma_wait(&bar_o, ph_o, p.err);

    // ---- the partial of this row over the prefix (the loads are warp-wide: every lane takes part) -----
    s_xch[tid] = l;
    __syncthreads();
    const float lt = l + s_xch[tid ^ kTcRows];
    const int64_t er = ((int64_t)h * p.Br + b) * p.R + r;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        float v[32];
        if (ntiles > 0) {
            tmem_ld32(tmem_o + lane_base + 32 * u, v);
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = 0.f;
        }
        if (live) {
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(p.ext_o + er * kHeadDim + col0 + 32 * u + c) =
                    make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
        }
    }
    if (live && half == 0) {
        p.ext_m[er] = m;
        p.ext_l[er] = lt;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

cudaError_t launch_prefix_tc(const PrefixTcParams& p, bool pdl, cudaStream_t s)
{
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(prefix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    dim3 grid((p.Br * p.R + kTcRows - 1) / kTcRows, p.Hkv);
    return launch_kernel(prefix_tc_kernel, grid, dim3(kTcThreads), kTcSmem, s, pdl, 0u, p);
}

}  // namespace fx
