// Split-KV decode attention on CUDA cores for sm_103a.
//
// One CTA (2 warps, 64 threads) = (row group of up to RB query rows, one split of the key sequence,
// one (b, KV head)).  The split is walked in tiles of 64 keys, one key per thread:
//   * K rows reach shared memory through the TMA engine: thread r issues one 256-byte
//     cp.async.bulk copy for key r of the tile (contiguous rows for the focal mode, gathered rows for
//     the sparse/prefix modes) into a row padded to 272 bytes, completing on an mbarrier.  With two
//     stages the next tile's rows are in flight while the current one is used.
//   * V rows go straight to registers: before waiting on K, each half-warp issues coalesced 16-byte
//     loads for its keys' V rows (lane `sub` holds dims [8*sub, 8*sub+8)).
//   * q.k is computed lane-per-key: each thread reads its own staged K row (the pad keeps the 32
//     rows of a warp on distinct banks) against the pre-scaled fp32 query rows broadcast from shared
//     memory -- no cross-lane reduction.  The softmax is kept online in base-2 units.
//   * p.v: half-warps take alternate keys, p is broadcast with one shuffle per (key, row).
// Partial (max, sum, unnormalised output) triples per split go to the workspace; the sparse/prefix
// modes merge them in the last-arriving CTA of each (b, h, row group), the focal mode in a separate
// combine kernel that also forms the per-token importance from the stored logits.
//
// Every mbarrier wait is bounded: on timeout the kernel sets FX_DEVERR_TIMEOUT, waits once more
// (bounded) for its own copies, and finishes without hanging.
//
// Attention and importance follow FastOCR (Methodology: Focal-Guided Pruning): focal layers attend
// over the full cache, the rest over the selected set; FastKV (2.A) for the causal query window;
// HPD-Parsing (parts 2 and 3) for the shared prefix + private suffix + causal draft sequence.
#include <math.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void unpack8(const uint4& w, float f[8])
{
    // bf16 -> fp32 is a 16-bit left shift of the pattern; element 2i is the low half of word i.
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
    f[4] = __uint_as_float(w.z << 16);
    f[5] = __uint_as_float(w.z & 0xffff0000u);
    f[6] = __uint_as_float(w.w << 16);
    f[7] = __uint_as_float(w.w & 0xffff0000u);
}

__device__ __forceinline__ uint4 ld_stream16(const uint16_t* ptr)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr));
    return r;
}

// 2^x with the hardware approximation (relative error about 2^-22, far inside the tolerances).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Bounded wait for phase `parity` of an mbarrier: never spins forever.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, unsigned* err)
{
    for (unsigned it = 0; it < kSpinLimit; ++it)
        if (mbar_try_wait(bar, parity)) return;
    atomicOr(err, FX_DEVERR_TIMEOUT);
    for (unsigned it = 0; it < kSpinLimit; ++it)   // give this CTA's own copies one more bounded chance
        if (mbar_try_wait(bar, parity)) return;
}

__device__ __forceinline__ void flag(unsigned* err, unsigned bit) { atomicOr(err, bit); }

// Thread-block-cluster helpers: rank, barrier, and loads from another CTA's shared memory.
__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_size()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_map(const void* p, unsigned rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Where the rows of one (b, h) key sequence live: sequence position -> K row and V row.
template <int MODE>
struct KeySource {
    const uint16_t* kb;   // main cache / prefix base for this (b, h)
    const uint16_t* vb;
    int64_t st;
    int kk;               // gathered positions (sparse idx / prefix idx)
    int tail_lo;          // sparse: first tail token
    int np, L;            // prefix: prefix rows, suffix rows
    const uint16_t* suf_k;
    const uint16_t* suf_v;
    int64_t suf_st;
    const uint16_t* dr_k;
    const uint16_t* dr_v;
    int64_t dr_si;
    bool gathered;        // prefix positions come from the index table
    int s0;

    __device__ __forceinline__ bool row(int pos, const int* s_tok, const uint16_t*& kp, const uint16_t*& vp) const
    {
        if (MODE == kModeFocal) {
            kp = kb + (int64_t)pos * st;
            vp = vb + (int64_t)pos * st;
            return true;
        }
        if (MODE == kModeSparse) {
            int t;
            if (pos < kk) {
                t = s_tok[pos - s0];
                if (t < 0) return false;
            } else {
                t = tail_lo + (pos - kk);
            }
            kp = kb + (int64_t)t * st;
            vp = vb + (int64_t)t * st;
            return true;
        }
        if (pos < np) {
            int t = pos;
            if (gathered) {
                t = s_tok[pos - s0];
                if (t < 0) return false;
            }
            kp = kb + (int64_t)t * st;
            vp = vb + (int64_t)t * st;
        } else if (pos < np + L) {
            const int64_t o = (int64_t)(pos - np) * suf_st;
            kp = suf_k + o;
            vp = suf_v + o;
        } else {
            const int64_t o = (int64_t)(pos - np - L) * dr_si;
            kp = dr_k + o;
            vp = dr_v + o;
        }
        return true;
    }
};

template <int MODE, int RB, bool CLUSTER>
__global__ void __launch_bounds__(kThreads) attn_decode_kernel(const AttnParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int nst = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* sK = smem + 128;
    float* q_s = reinterpret_cast<float*>(sK + (size_t)nst * kKStageBytes);
    int* s_tok = reinterpret_cast<int*>(q_s + RB * kHeadDim);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int hw = lane >> 4;
    const int sub = lane & 15;
    const int rg = blockIdx.x;
    const int split = blockIdx.y;
    const int bh = blockIdx.z;
    const int b = bh / p.Hkv;
    const int h = bh - b * p.Hkv;
    const int r0 = rg * RB;

    // ---- key sequence of this (b, h) ----------------------------------------------------------
    KeySource<MODE> src;
    int n_keys;
    src.kb = p.k + (int64_t)b * p.sb + (int64_t)h * p.sh;
    src.vb = p.v + (int64_t)b * p.sb + (int64_t)h * p.sh;
    src.st = p.st;
    src.kk = p.kk;
    src.tail_lo = p.tail_lo;
    src.gathered = p.idx != nullptr;
    src.np = 0;
    src.L = 0;
    int lim_tok = p.P;    // exclusive bound of a gathered index
    if (MODE == kModeFocal || MODE == kModeSparse) {
        int l = p.len[b];
        if (l < 0 || l > p.Tcap) {
            if (tid == 0) flag(p.err, FX_DEVERR_LEN);
            l = l < 0 ? 0 : p.Tcap;
        }
        n_keys = (MODE == kModeFocal) ? l : p.kk + max(0, l - p.tail_lo);
        lim_tok = l;
    } else {
        src.np = p.idx ? p.kk : p.P;
        const int o0 = p.suf_off[b];
        const int o1 = p.suf_off[b + 1];
        int L = 0;
        if (o0 < 0 || o1 < o0 || o1 > p.suf_rows) {
            if (tid == 0) flag(p.err, FX_DEVERR_OFFSETS);
        } else {
            L = o1 - o0;
            if (L > p.max_suffix) {
                if (tid == 0) flag(p.err, FX_DEVERR_OFFSETS);
                L = p.max_suffix;
            }
        }
        src.L = L;
        src.suf_k = p.suf_k + (int64_t)h * p.suf_sh + (int64_t)(L > 0 ? o0 : 0) * p.suf_st;
        src.suf_v = p.suf_v + (int64_t)h * p.suf_sh + (int64_t)(L > 0 ? o0 : 0) * p.suf_st;
        src.suf_st = p.suf_st;
        src.dr_k = p.dr_k + (int64_t)b * p.dr_sb + (int64_t)h * p.dr_sh;
        src.dr_v = p.dr_v + (int64_t)b * p.dr_sb + (int64_t)h * p.dr_sh;
        src.dr_si = p.dr_si;
        n_keys = src.np + L + p.Mq;
    }
    const int s0 = split * p.split_len;
    const int s1 = min(n_keys, s0 + p.split_len);
    src.s0 = s0;
    const int ntiles = s1 > s0 ? (s1 - s0 + kTile - 1) / kTile : 0;

    if (tid == 0) {
        mbar_init(smem_addr(&bars[0]), kThreads);
        mbar_init(smem_addr(&bars[1]), kThreads);
        mbar_init_fence();
    }
    // query rows, pre-scaled to base-2 logits
    for (int e = tid; e < RB * kHeadDim; e += kThreads) {
        const int r = e >> 7;
        const int c = e & (kHeadDim - 1);
        const int row = r0 + r;
        float v = 0.f;
        if (row < p.R) {
            const int gi = row / p.Mq;
            const int i = row - gi * p.Mq;
            const uint16_t qb = p.q[((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + c];
            v = __uint_as_float((uint32_t)qb << 16) * p.qscale;
        }
        q_s[e] = v;
    }
    // gathered token positions of this split, checked once
    if (MODE != kModeFocal && p.idx != nullptr) {
        const int32_t* irow = p.idx + (int64_t)bh * p.kk;
        const int hi = min(s1, p.kk);
        for (int pos = s0 + tid; pos < hi; pos += kThreads) {
            int t = __ldg(irow + pos);
            if (t < 0 || t >= lim_tok) {
                flag(p.err, FX_DEVERR_INDEX);
                t = -1;
            }
            s_tok[pos - s0] = t;
        }
    }
    __syncthreads();

    int lim[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int row = r0 + r;
        const int i = row - (row / p.Mq) * p.Mq;
        if (row >= p.R)
            lim[r] = -1;   // padding row: sees nothing
        else if (MODE == kModeFocal)
            lim[r] = p.q_pos0 >= 0 ? p.q_pos0 + i : 0x7fffffff;
        else if (MODE == kModePrefix)
            lim[r] = src.np + src.L + i;   // draft row j is visible iff j <= i
        else
            lim[r] = 0x7fffffff;
    }

    // thread r stages K row r of a tile (one 256-byte bulk copy) or zero-fills it
    auto issue = [&](int tile, int stage) {
        const int pos = s0 + tile * kTile + tid;
        const uint16_t* kp = src.kb;
        const uint16_t* vp = src.vb;
        const bool ok = pos < s1 && src.row(pos, s_tok, kp, vp);
        unsigned char* dst = sK + (size_t)stage * kKStageBytes + (size_t)tid * kKPitch;
        const uint32_t bar = smem_addr(&bars[stage]);
        fence_proxy_async();
        if (ok) {
            mbar_arrive_expect_tx(bar, kRowBytes);
            bulk_g2s(smem_addr(dst), kp, kRowBytes, bar);
        } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int c = 0; c < kRowBytes / 16; ++c) d4[c] = make_uint4(0u, 0u, 0u, 0u);
            mbar_arrive(bar);
        }
    };

    float m[RB], lsum[RB], o[RB][8];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        m[r] = -INFINITY;
        lsum[r] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][e] = 0.f;
    }
    uint32_t phase_bits = 0u;   // bit s: parity of the next completion of stage s

    if (ntiles > 0) issue(0, 0);
    if (ntiles > 1 && nst > 1) issue(1, 1);

    for (int tile = 0; tile < ntiles; ++tile) {
        const int stage = nst > 1 ? (tile & 1) : 0;
        const int base = s0 + tile * kTile;

        // V rows of this warp's 32 keys, straight to registers (half-warp per key)
        uint4 vr[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int pos = base + warp * 32 + 2 * i + hw;
            const uint16_t* kp;
            const uint16_t* vp;
            const bool ok = pos < s1 && src.row(pos, s_tok, kp, vp);
            vr[i] = ok ? ld_stream16(vp + sub * 8) : make_uint4(0u, 0u, 0u, 0u);
        }

        mbar_wait(smem_addr(&bars[stage]), (phase_bits >> stage) & 1u, p.err);
        phase_bits ^= 1u << stage;

        // q.k, one key per lane
        const int kpos = base + tid;
        bool kval = kpos < s1;
        if (MODE == kModeSparse && kval && kpos < p.kk) kval = s_tok[kpos - s0] >= 0;
        if (MODE == kModePrefix && kval && src.gathered && kpos < src.np) kval = s_tok[kpos - s0] >= 0;
        const unsigned char* krow = sK + (size_t)stage * kKStageBytes + (size_t)tid * kKPitch;
        float acc[RB][4];   // four independent FMA chains per row
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[r][j] = 0.f;
#pragma unroll 4
        for (int c = 0; c < kHeadDim / 8; ++c) {
            float kf[8];
            unpack8(*reinterpret_cast<const uint4*>(krow + c * 16), kf);
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float4 qa = *reinterpret_cast<const float4*>(q_s + r * kHeadDim + c * 8);
                const float4 qb = *reinterpret_cast<const float4*>(q_s + r * kHeadDim + c * 8 + 4);
                acc[r][0] = fmaf(qa.x, kf[0], acc[r][0]);
                acc[r][1] = fmaf(qa.y, kf[1], acc[r][1]);
                acc[r][2] = fmaf(qa.z, kf[2], acc[r][2]);
                acc[r][3] = fmaf(qa.w, kf[3], acc[r][3]);
                acc[r][0] = fmaf(qb.x, kf[4], acc[r][0]);
                acc[r][1] = fmaf(qb.y, kf[5], acc[r][1]);
                acc[r][2] = fmaf(qb.z, kf[6], acc[r][2]);
                acc[r][3] = fmaf(qb.w, kf[7], acc[r][3]);
            }
        }
        float pr[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r)
            pr[r] = (kval && kpos <= lim[r]) ? (acc[r][0] + acc[r][1]) + (acc[r][2] + acc[r][3]) : -INFINITY;

        if (MODE == kModeFocal && p.logits != nullptr && kpos < s1) {
#pragma unroll
            for (int r = 0; r < RB; ++r)
                if (r0 + r < p.R) p.logits[(int64_t)(bh * p.R + r0 + r) * p.Tcap + kpos] = pr[r];
        }

        // online softmax (warp-uniform running max)
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float cm = pr[r];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, off));
            const float mn = fmaxf(m[r], cm);
            const float ms = (mn == -INFINITY) ? 0.f : mn;
            const float alpha = fast_exp2(m[r] - ms);
            m[r] = mn;
            lsum[r] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[r][e] *= alpha;
            pr[r] = fast_exp2(pr[r] - ms);
            lsum[r] += pr[r];
        }

        // p.v: half-warp hw takes keys 2i + hw of this warp
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float vf[8];
            unpack8(vr[i], vf);
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float pk = __shfl_sync(kFull, pr[r], 2 * i + hw);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[r][e] = fmaf(pk, vf[e], o[r][e]);
            }
        }

        __syncthreads();   // both warps are done with this K stage
        if (tile + nst < ntiles) issue(tile + nst, stage);
    }

    // reduce within the warp: lsum over all lanes, o over the two half-warps
#pragma unroll
    for (int r = 0; r < RB; ++r) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lsum[r] += __shfl_xor_sync(kFull, lsum[r], off);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][e] += __shfl_xor_sync(kFull, o[r][e], 16);
    }

    // ---- combine the two warps into one partial per row (the K stages are free now) -----------
    __shared__ float sm_m[kWarps][RB];
    __shared__ float sm_l[kWarps][RB];
    float* sm_o = reinterpret_cast<float*>(sK);   // [kWarps][RB][128]
    if (lane < 16) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float4* dst = reinterpret_cast<float4*>(sm_o + (warp * RB + r) * kHeadDim + sub * 8);
            dst[0] = make_float4(o[r][0], o[r][1], o[r][2], o[r][3]);
            dst[1] = make_float4(o[r][4], o[r][5], o[r][6], o[r][7]);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            sm_m[warp][r] = m[r];
            sm_l[warp][r] = lsum[r];
        }
    }
    __syncthreads();

    // this CTA's partial: c_m / c_l / c_o (also read by the other CTAs of the cluster)
    __shared__ float c_m[RB];
    __shared__ float c_l[RB];
    __shared__ __align__(16) float c_o[RB][kHeadDim];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][r]);
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float sc[kWarps];
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            sc[w] = fast_exp2(sm_m[w][r] - Ms);
            Ls = fmaf(sm_l[w][r], sc[w], Ls);
        }
        for (int c = tid; c < kHeadDim; c += kThreads) {
            float O = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) O = fmaf(sm_o[(w * RB + r) * kHeadDim + c], sc[w], O);
            c_o[r][c] = O;
        }
        if (tid == 0) {
            c_m[r] = M;
            c_l[r] = Ls;
        }
    }
    const int nr = min(RB, p.R - r0);   // rows of this row group that exist

    if (CLUSTER) {
        // every split of this (b, h, row group) is one CTA of the cluster: merge through distributed
        // shared memory, each CTA producing a slice of the output rows
        cluster_sync();
        const unsigned cs = cluster_size();
        const unsigned me = cluster_rank();
        for (int e = (int)me * kThreads + tid; e < nr * kHeadDim; e += (int)cs * kThreads) {
            const int r = e >> 7;
            const int c = e & (kHeadDim - 1);
            float M = -INFINITY;
            for (unsigned q = 0; q < cs; ++q) M = fmaxf(M, ld_cluster(cluster_map(&c_m[r], q)));
            const float Ms = (M == -INFINITY) ? 0.f : M;
            float Ls = 0.f, O = 0.f;
            for (unsigned q = 0; q < cs; ++q) {
                const float w = fast_exp2(ld_cluster(cluster_map(&c_m[r], q)) - Ms);
                Ls = fmaf(ld_cluster(cluster_map(&c_l[r], q)), w, Ls);
                O = fmaf(ld_cluster(cluster_map(&c_o[r][c], q)), w, O);
            }
            const int row = r0 + r;
            const int gi = row / p.Mq;
            const int i = row - gi * p.Mq;
            p.out[((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + c] = Ls > 0.f ? O / Ls : 0.f;
        }
        cluster_sync();   // keep every CTA's shared memory alive until all reads are done
        return;
    }

    __syncthreads();
    for (int r = 0; r < nr; ++r) {
        const int64_t pi = (int64_t)(bh * p.R + r0 + r) * p.nsplit + split;
        for (int c = tid; c < kHeadDim; c += kThreads) p.part_o[pi * kHeadDim + c] = c_o[r][c];
        if (tid == 0) {
            p.part_m[pi] = c_m[r];
            p.part_l[pi] = c_l[r];
        }
    }

    if (MODE == kModeFocal) return;

    // ---- last-arriving CTA of this (b, h, row group) merges the splits ------------------------
    __shared__ unsigned s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&p.counters[bh * p.nrg + rg], 1u);
        s_last = (prev == (unsigned)(p.nsplit - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (s_last == 0u) return;
    __threadfence();
    for (int r = 0; r < nr; ++r) {
        const int row = r0 + r;
        const int64_t base = (int64_t)(bh * p.R + row) * p.nsplit;
        float M = -INFINITY;
        for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, __ldcg(p.part_m + base + s));
        const float Ms = (M == -INFINITY) ? 0.f : M;
        const int gi = row / p.Mq;
        const int i = row - gi * p.Mq;
        float* orow = p.out + ((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7);
        for (int c = tid; c < kHeadDim; c += kThreads) {
            float Ls = 0.f, O = 0.f;
            for (int s = 0; s < p.nsplit; ++s) {
                const float sc = fast_exp2(__ldcg(p.part_m + base + s) - Ms);
                Ls = fmaf(__ldcg(p.part_l + base + s), sc, Ls);
                O = fmaf(__ldcg(p.part_o + (base + s) * kHeadDim + c), sc, O);
            }
            orow[c] = Ls > 0.f ? O / Ls : 0.f;
        }
    }
    if (tid == 0) p.counters[bh * p.nrg + rg] = 0u;
}

// Focal combine: merge split partials into the output rows and form the importance scores
//   s_j = sum_r exp2(t_rj - M_r) / Z_r   over the group's rows r, for cand_lo <= j < cand_hi.
__global__ void __launch_bounds__(256) focal_combine_kernel(const FocalCombineParams p)
{
    const int bh = blockIdx.y;
    const int b = bh / p.Hkv;
    const int h = bh - b * p.Hkv;
    __shared__ float sM[kMaxRows];
    __shared__ float sInvZ[kMaxRows];
    for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
        const int64_t base = (int64_t)(bh * p.R + r) * p.nsplit;
        float M = -INFINITY;
        for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, p.part_m[base + s]);
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float Z = 0.f;
        for (int s = 0; s < p.nsplit; ++s) Z = fmaf(p.part_l[base + s], fast_exp2(p.part_m[base + s] - Ms), Z);
        sM[r] = Ms;
        sInvZ[r] = Z > 0.f ? 1.f / Z : 0.f;
    }
    __syncthreads();

    if (blockIdx.x == 0 && p.out != nullptr) {
        for (int e = threadIdx.x; e < p.R * kHeadDim; e += blockDim.x) {
            const int r = e >> 7;
            const int c = e & (kHeadDim - 1);
            const int64_t base = (int64_t)(bh * p.R + r) * p.nsplit;
            float O = 0.f;
            for (int s = 0; s < p.nsplit; ++s)
                O = fmaf(p.part_o[(base + s) * kHeadDim + c], fast_exp2(p.part_m[base + s] - sM[r]), O);
            const int gi = r / p.Mq;
            const int i = r - gi * p.Mq;
            p.out[((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + c] = O * sInvZ[r];
        }
    }

    if (p.scores != nullptr) {
        int lenb = p.len[b];
        lenb = lenb < 0 ? 0 : (lenb > p.Tcap ? p.Tcap : lenb);
        const int ncand = p.cand_hi - p.cand_lo;
        float* srow = p.scores + (int64_t)bh * ncand;
        const float* lrow = p.logits + (int64_t)bh * p.R * p.Tcap;
        for (int jj = blockIdx.x * blockDim.x + threadIdx.x; jj < ncand; jj += gridDim.x * blockDim.x) {
            const int j = p.cand_lo + jj;
            float s = 0.f;
            if (j < lenb) {
                for (int r = 0; r < p.R; ++r)
                    s = fmaf(fast_exp2(__ldcs(lrow + (int64_t)r * p.Tcap + j) - sM[r]), sInvZ[r], s);
            }
            srow[jj] = s;
        }
    }
}

template <int MODE, int RB, bool CLUSTER>
cudaError_t launch_one(const AttnParams& p, cudaStream_t s)
{
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = attn_decode_kernel<MODE, RB, CLUSTER>;
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)attn_smem_bytes(2, RB, kMaxSplitTokens));
        if (e != cudaSuccess) return e;
        if (CLUSTER) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        configured = dev;
    }
    const size_t smem = attn_smem_bytes(p.stages, RB, (MODE != kModeFocal && p.idx != nullptr) ? p.split_len : 0);
    dim3 grid(p.nrg, p.nsplit, p.B * p.Hkv);
    if (!CLUSTER) {
        kern<<<grid, kThreads, smem, s>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.nsplit;   // every split of one (b, h, row group)
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int MODE, bool CLUSTER>
cudaError_t launch_mode(const AttnParams& p, int rb, cudaStream_t s)
{
    switch (rb) {
    case 1: return launch_one<MODE, 1, CLUSTER>(p, s);
    case 2: return launch_one<MODE, 2, CLUSTER>(p, s);
    case 4: return launch_one<MODE, 4, CLUSTER>(p, s);
    default: return launch_one<MODE, 8, CLUSTER>(p, s);
    }
}

}  // namespace

cudaError_t launch_attn_partial(const AttnParams& p, int mode, int rb, cudaStream_t s)
{
    if (mode == kModeFocal) return launch_mode<kModeFocal, false>(p, rb, s);
    const bool cl = p.nsplit <= kMaxClusterSplits;
    if (mode == kModeSparse)
        return cl ? launch_mode<kModeSparse, true>(p, rb, s) : launch_mode<kModeSparse, false>(p, rb, s);
    return cl ? launch_mode<kModePrefix, true>(p, rb, s) : launch_mode<kModePrefix, false>(p, rb, s);
}

cudaError_t launch_focal_combine(const FocalCombineParams& p, cudaStream_t s)
{
    const int ncand = p.scores ? (p.cand_hi - p.cand_lo) : 0;
    int gx = (ncand + 1023) / 1024;
    if (gx < 1) gx = 1;
    if (gx > 256) gx = 256;
    dim3 grid(gx, p.B * p.Hkv);
    focal_combine_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace fx
