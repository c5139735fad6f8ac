// Dense shared-prefix attention on the tensor cores of sm_103a (tcgen05, accumulators in tensor memory).
//
// HPD-Parsing (part 2, shared-prefix KV reuse; part 3, parallel verification of drafted tokens): every
// branch attends over the same prefix rows (up to its fork position) before its own suffix and drafts.
// Per KV head the query rows of all branches (Br x R of them) therefore meet one shared set of keys --
// a real matrix product, which this kernel runs as 128 x 128 tiles on the tensor cores:
//   S = Q K^T       (M = 128 query rows, N = 128 prefix keys, K = 128 dims)   smem x smem -> tensor memory
//   O += P V        (M = 128 query rows, N = 128 dims, K = 128 prefix keys)   tensor memory x smem -> tensor memory
// in one pass with an online softmax (P = exp2(S - m) against a running maximum m that moves only by
// more than a fixed slack, so O is rescaled rarely), P split into bf16 hi + lo parts (two products) so
// the probabilities keep about 16 bits.  Eight softmax warps own the 128 query rows, two threads per
// row, each for half of the keys of a tile and half of O: they read their S columns from tensor
// memory, trade the row maximum with the partner warp, and write P back into tensor memory (two
// buffers), where the P V product takes it as its A operand.  A ninth warp issues the products when
// mbarriers say the softmax warps have published their operands.  Q and K tiles are K-major operands
// with the 128-byte swizzle; V tiles are copied as they are stored (keys x dims) into the same
// swizzled layout and used as an MN-major operand, so nothing is transposed.  K and V are double
// buffered in shared memory: the next tile's Q K^T and the previous tile's P V run on the tensor cores
// while this tile's softmax runs on the softmax warps.
// The result per row is a partial (m, l, O) over the prefix, which the verify kernel folds into its
// merge of the suffix and draft keys.
#include <cuda_bf16.h>
#include <stdint.h>

#include "fx_internal.h"
#include "tc_ptx.cuh"

namespace fx {
namespace {

constexpr int kTcRows = 128;                       // query rows per CTA (one tensor-memory lane each)
constexpr int kTcKeys = 128;                       // prefix keys per tile
constexpr int kTcSoftmax = 256;                    // softmax threads: two per query row (warps 0..7)
constexpr int kTcThreads = kTcSoftmax + 32;        // and one warp that issues the products
constexpr int kTileBytes = kTcRows * kHeadDim * 2;  // one 128 x 128 bf16 operand tile
// tensor-memory columns: S, O, and P of even and odd tiles (bf16 pairs: 64 columns hi, then 64 lo)
constexpr int kTmemCols = 512;
constexpr int kColS = 0, kColO = 128, kColP0 = 256, kColP1 = 384;
// [Q | K even | K odd | V even | V odd] swizzled tiles and slack to align to 1024 bytes
constexpr size_t kTcSmem = 5 * (size_t)kTileBytes + 1024;

// S (tensor memory) = Q (smem tile) x K (smem tile)^T over the 128 dims, as 8 products of K = 16.
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint32_t q_tile, uint32_t k_tile)
{
    constexpr uint32_t idesc = idesc_bf16(128, 128, false);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (uint32_t)((ks >> 2) * kTileBytes / 2 + (ks & 3) * 32);
        const uint64_t da = sdesc(q_tile + off);
        const uint64_t db = sdesc(k_tile + off);
        const uint32_t acc = ks > 0 ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(da), "l"(db), "r"(idesc), "r"(acc));
    }
}

// O (tensor memory) (+)= P (tensor memory, bf16 pairs) x V (smem tile, MN-major) over the 128 keys.
__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_tile, bool accumulate)
{
    constexpr uint32_t idesc = idesc_bf16(128, 128, true);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint64_t db = sdesc(v_tile + ks * 2048, kTileBytes / 2);   // 16 keys = two 8-row groups
        const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(p_tmem + 8 * ks), "l"(db), "r"(idesc), "r"(acc));
    }
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

// Paired fp32 arithmetic (one instruction for two lanes of a pair) and a three-input maximum.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Arrive on a CTA mbarrier (release: this thread's earlier shared-memory and tensor-memory work is
// ordered before the waiter's acquire).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bounded wait (acquire) for the phase of a CTA mbarrier with the given parity; flags a timeout.
__device__ __forceinline__ void mbar_wait(uint64_t* bar, unsigned parity, unsigned* err)
{
    unsigned spins = 0, done = 0;
    while (!done) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (!done && ++spins == kSpinLimit) {
            atomicOr(err, FX_DEVERR_TIMEOUT);
            break;
        }
    }
}

// Barrier of the two softmax warps that share a row quarter (warps w and w + 4): named barrier 1 + w.
__device__ __forceinline__ void pair_sync(int warp)
{
    asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1) prefix_tc_kernel(const PrefixTcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char* sQ = base;
    auto sK = [&](int x) { return base + (1 + x) * kTileBytes; };   // K tiles of even / odd tiles
    auto sV = [&](int x) { return base + (3 + x) * kTileBytes; };   // V tiles of even / odd tiles
    __shared__ __align__(8) uint64_t bar_s;      // S of the current tile is in tensor memory (commit)
    __shared__ __align__(8) uint64_t bar_o;      // O += P V of the last issued tile is done (commit)
    __shared__ __align__(8) uint64_t bar_sgo;    // softmax threads: S read, next K published
    __shared__ __align__(8) uint64_t bar_pgo;    // softmax threads: P written, V published
    __shared__ uint32_t s_tmem;
    __shared__ int s_lim_max;
    __shared__ float s_xch[2][kTcSoftmax];       // the two halves of a row trade their maxima (per tile parity)
    __shared__ float s_lsum[kTcSoftmax];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const bool softmax = tid < kTcSoftmax;       // warps 0..7; warp 8 issues the products
    const int lrow = tid & (kTcRows - 1);        // query row within the tile = tensor-memory lane
    const int half = (tid >> 7) & 1;             // this thread's 64 keys of each tile and 64 dims of O
    const int col0 = half * 64;
    const int h = blockIdx.y;
    const int rows_total = p.Br * p.R;
    const int row = blockIdx.x * kTcRows + lrow;
    const bool live = softmax && row < rows_total;
    const int b = live ? row / p.R : 0;
    const int r = live ? row - b * p.R : 0;

    griddep_wait();   // the queries may come from the kernel just before
    // The verify kernel launched right after this one reads its lengths, offsets and K/V rows before its
    // own dependency wait (fx_shared_prefix_decode launches it that way whatever the caller's flags).
    // That is sound only because this trigger comes after this kernel's wait above: when the verify
    // kernel starts, everything enqueued before this kernel has finished.  Do not move it earlier.
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
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&bar_sgo)), "r"(kTcSoftmax));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&bar_pgo)), "r"(kTcSoftmax));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // this row's query into the Q tile (zero past the last row); each half copies 64 dims
    if (softmax) {
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
    if (softmax) atomicMax(&s_lim_max, lim);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int ntiles = (s_lim_max + kTcKeys - 1) / kTcKeys;
    const uint16_t* kb = p.pk + (int64_t)h * p.p_sh;
    const uint16_t* vb = p.pv + (int64_t)h * p.p_sh;

    // Tiles t = 0 .. ntiles-1 (x = t & 1 picks the K, V and P buffers): K(t) -> sK(x), V(t) -> sV(x),
    // S(t) = Q K(t)^T -> tensor-memory S, P(t) -> tensor-memory P[x], O += P(t) V(t).  Warp 8 issues the
    // products, each when the softmax warps say its operands are ready (bar_sgo: everyone has read S(t)
    // and published K(t+1); bar_pgo: everyone has written P(t) and published V(t)); the softmax warps
    // wait only on the products' completion barriers and, for the row maximum, on their partner warp.
    if (!softmax) {
        const int lane = tid & 31;
        if (ntiles > 0) {
            mbar_wait(&bar_sgo, 0u, p.err);   // Q and K(0) published
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (lane == 0) {
                mma_qk(tmem + kColS, smem_addr(sQ), smem_addr(sK(0)));
                mma_commit(&bar_s);
            }
        }
        for (int t = 0; t < ntiles; ++t) {
            const int x = t & 1;
            if (t + 1 < ntiles) {
                mbar_wait(&bar_sgo, (unsigned)(t + 1) & 1u, p.err);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (lane == 0) {
                    mma_qk(tmem + kColS, smem_addr(sQ), smem_addr(sK(x ^ 1)));
                    mma_commit(&bar_s);
                }
            }
            mbar_wait(&bar_pgo, (unsigned)t & 1u, p.err);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (lane == 0) {
                const uint32_t col_p = x ? kColP1 : kColP0;
                mma_pv(tmem + kColO, tmem + col_p, smem_addr(sV(x)), t > 0);
                mma_pv(tmem + kColO, tmem + col_p + 64, smem_addr(sV(x)), true);
                mma_commit(&bar_o);
            }
        }
    } else {
        // Thread tid copies 16-byte chunk (tid & 15) of keys key0 + 16 i (i = 0..7) of every tile: the
        // swizzled offsets of those rows are 2048 i apart, the source rows 16 i * p_st elements apart.
        const int key0 = tid >> 4;
        const int chunk = tid & 15;
        const uint32_t soff0 = sw128(key0, 8 * chunk, kTcKeys);
        const int64_t goff0 = (int64_t)key0 * p.p_st + 8 * chunk;
        const int64_t gstep = (int64_t)16 * p.p_st;
        // one commit group per call, empty when the tile does not exist, so the group counts stay fixed:
        // K(0), V(0), K(1) before the loop, then K(t+2) and V(t+1) per tile
        auto load_tile = [&](unsigned char* dst, const uint16_t* src, int t) {
            if (t < ntiles) {
                const int j0 = t * kTcKeys;
                const uint16_t* g = src + (int64_t)j0 * p.p_st + goff0;
                const uint32_t d0 = smem_addr(dst) + soff0;
                if (j0 + kTcKeys <= p.P) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) cp16(d0 + 2048 * i, g + i * gstep);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (j0 + key0 + 16 * i < p.P)
                            cp16(d0 + 2048 * i, g + i * gstep);
                        else
                            *reinterpret_cast<uint4*>(dst + soff0 + 2048 * i) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // hand shared-memory operands (and the tensor-memory work before) to the issuing warp
        auto publish = [&](uint64_t* bar) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(bar);
        };

        // Online softmax: a row's running maximum m moves only when a tile's maximum exceeds it by more
        // than kMaxSlack (log2 units); O in tensor memory is then rescaled by the row's threads, and
        // P = exp2(s - m) stays below 2^kMaxSlack.
        float m = -INFINITY;
        float l = 0.f;   // this half's share of the row sum
        if (ntiles > 0) {
            load_tile(sK(0), kb, 0);
            load_tile(sV(0), vb, 0);
            load_tile(sK(1), kb, 1);
            asm volatile("cp.async.wait_group 2;" ::: "memory");   // K(0)
            publish(&bar_sgo);
        }
        for (int t = 0; t < ntiles; ++t) {
            const int x = t & 1;
            const int j0 = t * kTcKeys;
            const uint32_t col_p = x ? kColP1 : kColP0;
            // (b) this half's 64 logits of S(t); then K(t+2) into S(t)'s K buffer, and K(t+1) published
            // together with the end of this thread's reads of S
            mma_wait_parity(&bar_s, (unsigned)t & 1u, p.err);
            float sv[2][32];
            tmem_ld32(tmem + lane_base + kColS + col0, sv[0]);
            tmem_ld32(tmem + lane_base + kColS + col0 + 32, sv[1]);
            load_tile(sK(x), kb, t + 2);
            if (t + 1 < ntiles) {
                if (t == 0)
                    asm volatile("cp.async.wait_group 1;" ::: "memory");   // K(1)
                else
                    asm volatile("cp.async.wait_group 2;" ::: "memory");   // K(t+1); V(t), K(t+2) may fly
                publish(&bar_sgo);
            }
            // (c) the row's maximum over the tile: the two halves trade theirs
            const int nv = lim - (j0 + col0);   // keys of this half that the row sees
            const bool full = nv >= 64;
            float mt = -INFINITY;
            if (full && p.qscale > 0.f) {   // max of the raw logits, scaled once
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 2) mt = max3(mt, sv[u][jj], sv[u][jj + 1]);
                mt *= p.qscale;
            } else {
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (32 * u + jj < nv) mt = fmaxf(mt, sv[u][jj] * p.qscale);
            }
            s_xch[x][tid] = mt;
            pair_sync(warp);
            mt = fmaxf(mt, s_xch[x][tid ^ kTcRows]);
            const bool grow = mt > m + kMaxSlack;   // also when m is still -inf and the tile has keys
            const float mnew = grow ? mt : m;
            // (d) a moved maximum rescales O, once P(t-1) V(t-1) is done
            if (t > 0 && __any_sync(0xffffffffu, grow)) {   // tensor-memory access is warp-wide
                mma_wait_parity(&bar_o, (unsigned)(t - 1) & 1u, p.err);
                const float a = !grow ? 1.f : (m == -INFINITY ? 0.f : exp2_approx(m - mnew));
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float v[32];
                    uint32_t w[32];
                    tmem_ld32(tmem + lane_base + kColO + col0 + 32 * u, v);
#pragma unroll
                    for (int c = 0; c < 32; ++c) w[c] = __float_as_uint(v[c] * a);
                    tmem_st32(tmem + lane_base + kColO + col0 + 32 * u, w);
                }
                l *= a;
            }
            m = mnew;
            const float ms = (m == -INFINITY) ? 0.f : m;
            // (e) P(t) = exp2(s - m) as bf16 pairs (key 2i in the low half), hi and lo parts, l += sum P;
            // the P buffer of tile t was last read by P(t-2) V(t-2), finished before (f) of tile t-1
            {
                uint32_t ph[32], pl[32];
                float2 l2 = make_float2(0.f, 0.f);
                auto pair = [&](int k2, float p0, float p1) {
                    const float2 pp = make_float2(p0, p1);
                    l2 = add2(l2, pp);
                    __nv_bfloat162 hv = __floats2bfloat162_rn(p0, p1);
                    ph[k2] = *reinterpret_cast<uint32_t*>(&hv);
                    const float2 lo = sub2(pp, make_float2(__low2float(hv), __high2float(hv)));
                    pl[k2] = pack2_bf16(lo.x, lo.y);
                };
                const float2 qs2 = make_float2(p.qscale, p.qscale);
                const float2 nms2 = make_float2(-ms, -ms);
                if (full) {
#pragma unroll
                    for (int k2 = 0; k2 < 32; ++k2) {
                        const int e0 = 2 * k2;
                        const float2 x2 =
                            fma2(make_float2(sv[e0 >> 5][e0 & 31], sv[e0 >> 5][(e0 & 31) + 1]), qs2, nms2);
                        pair(k2, exp2_approx(x2.x), exp2_approx(x2.y));
                    }
                } else {
#pragma unroll
                    for (int k2 = 0; k2 < 32; ++k2) {
                        const int e0 = 2 * k2;
                        const float2 x2 =
                            fma2(make_float2(sv[e0 >> 5][e0 & 31], sv[e0 >> 5][(e0 & 31) + 1]), qs2, nms2);
                        pair(k2, e0 < nv ? exp2_approx(x2.x) : 0.f, e0 + 1 < nv ? exp2_approx(x2.y) : 0.f);
                    }
                }
                l += l2.x + l2.y;
                tmem_st32(tmem + lane_base + col_p + half * 32, ph);
                tmem_st32(tmem + lane_base + col_p + 64 + half * 32, pl);
            }
            // (f) P(t-1) V(t-1) done (issued a tile ago): its V buffer takes V(t+1); V(t) has landed;
            // P(t) and V(t) go to the issuing warp
            if (t > 0) mma_wait_parity(&bar_o, (unsigned)(t - 1) & 1u, p.err);
            asm volatile("cp.async.wait_group 1;" ::: "memory");   // V(t); K(t+2) may fly
            load_tile(sV(x ^ 1), vb, t + 1);
            publish(&bar_pgo);
        }
        if (ntiles > 0) mma_wait_parity(&bar_o, (unsigned)(ntiles - 1) & 1u, p.err);

        // ---- the partial of this row over the prefix (the loads are warp-wide: every lane takes part) --
        s_lsum[tid] = l;
        pair_sync(warp);
        const float lt = l + s_lsum[tid ^ kTcRows];
        const int64_t er = ((int64_t)h * p.Br + b) * p.R + r;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float v[32];
            if (ntiles > 0) {
                tmem_ld32(tmem + lane_base + kColO + col0 + 32 * u, v);
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
