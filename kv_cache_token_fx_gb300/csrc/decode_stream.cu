// Streaming sparse decode attention for sm_103a: the decode-shaped calls of fx_sparse_gqa_decode (one
// query position, at most 8 query rows per KV head).
//
// One CTA = one (sequence b, KV head h, split of the key sequence), with two warp roles:
//   * NP producer warps stage the split's 16-key sub-tiles (16 K rows and 16 V rows of 256 bytes,
//     gathered through the index list or taken from the dense tail) into a CTA-wide ring of S slots
//     with 16-byte cp.async, producer p taking sub-tiles j = p, p + NP, ... (so it owns the slots
//     s = p mod NP of the ring).  Each slot has a "full" mbarrier that every producer lane arrives on
//     asynchronously (cp.async.mbarrier.arrive.noinc: the arrival fires when that lane's copies have
//     landed) and an "empty" mbarrier the consuming warp arrives on once it has read the slot.  A
//     rejected row is zero-filled by the copy itself (source size 0).  The producer never publishes
//     anything with a plain store: a release arrival after outstanding cp.async would wait for them.
//     Index entries are loaded a full ring ahead of their use, so the producer never waits on them;
//     each producer keeps at most S / NP sub-tiles (S / NP * 8 KB) in flight, below the per-warp
//     limit of outstanding cp.async beyond which issuing stalls.
//   * C consumer warps take the sub-tiles round-robin (sub-tile j goes to warp j mod C), wait for its
//     slot, and fold it into their own online-softmax state with mma.sync m16n8k16 in the keys-on-M
//     layout: S^T = K Q^T (16 keys x 8 query rows), O^T += V^T P^T with P^T moved into the B operand by
//     movmatrix.trans and P split into bf16 hi + lo parts (two MMAs, ~16-bit probabilities).  A
//     consumer tells valid rows from rejected ones with the same index test as the producer, on index
//     entries it loads one sub-tile ahead.
// The ring decouples the bytes in flight (S slots, 8 KB each) from the warps doing math.
//
// Why this shape: a decode call reads 20-30 MB in a few microseconds, so the fixed parts of a launch
// (index loads, the first HBM round trip, the merge) are a large share of it.  The host picks about
// one CTA per SM per call and a ring that lets two CTAs share an SM; the next layer's call (launched as
// a programmatic dependent) is then resident while this one finishes, and its producer warps fill
// their rings -- index loads and K/V copies -- during this call's last round trip and merge.  Only its
// query rows wait for this call.  The next call is released once this call's producers have issued
// every copy: released earlier, its ring fill would queue in HBM ahead of this call's own refills.
//
// Merge: the warps' partials (max, sum, unnormalised output) are combined in shared memory with per-row
// weights; the splits of one (b, h) form a thread-block cluster and the others push their combined
// partial into CTA 0 with st.async (completing bytes on CTA 0's mbarrier), which writes the output.
//
// What is computed follows FastOCR (Methodology: Focal-Guided Pruning: a non-focal layer attends only
// to the pruned set; the softmax is renormalised over that set) and FastKV (2.B: decoding over the
// retained entries).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "attn_ptx.cuh"
#include "fx_internal.h"

namespace fx {
namespace {

constexpr int kRows = 8;                       // query rows of the keys-on-M tile
constexpr int kOPitch = kHeadDim + 8;          // warp-partial rows in the epilogue (floats)

// 16-byte cp.async that copies `bytes` (16 or 0) bytes and zero-fills the rest of the 16.
__device__ __forceinline__ void cp_async16_fill(uint32_t dst, const void* src, unsigned bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
// Arrival on `bar` once every cp.async this thread issued before it has landed; the barrier's initial
// count includes this arrival.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Arrivals without release semantics (nothing is published through them; a release arrival would also
// wait for this thread's outstanding cp.async writes).
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint64_t* bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
// TMA tile load of the box at (c0, c1, c2, c3) of a 4-D tensor map into shared memory; its bytes
// complete on `bar`.  c0 (the element column) must be a multiple of 8 (16 bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
        : "memory");
}
// Byte offset of 16-byte chunk c (0..15) of row `row` (0..15) inside a staged K or V sub-tile: the layout
// a TMA box of 16 rows x 64 columns with the 128-byte swizzle writes -- columns 0-63 in the first 2 KB,
// 64-127 in the next, 128 bytes per row, chunk index XORed with (row % 8) -- so that the 8 rows an
// ldmatrix reads at one chunk fall on 8 bank groups.  Gathered rows are copied into the same layout.
__device__ __forceinline__ uint32_t tile_off(int row, int c)
{
    return (uint32_t)(((c >> 3) << 11) + (row << 7) + (((c & 7) ^ (row & 7)) << 4));
}
constexpr int kHalfTile = kSub * 128;   // bytes of one 16-row x 64-column box

template <int C, int NP, bool CLUSTER>
__global__ void __launch_bounds__(32 * (C + NP), 2)
    stream_decode_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // the ring starts on a 1024-byte boundary (the period of the 128-byte swizzle)
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages;                                               // ring slots (a multiple of NP)
    unsigned char* ring = smem;                                           // [S][K 16 rows | V 16 rows]
    unsigned char* sQ = smem + (size_t)S * kSubBytes;                     // [8][kPitch] bf16
    float* s_recv = reinterpret_cast<float*>(sQ + kRows * kPitch);        // pushed partials (cluster CTA 0)
    __shared__ __align__(8) uint64_t full_bar[kStreamMaxSlots];
    __shared__ __align__(8) uint64_t empty_bar[kStreamMaxSlots];
    __shared__ __align__(8) uint64_t merge_bar;
    __shared__ __align__(8) uint64_t stall_bar;   // testing: a barrier nothing arrives on
    __shared__ float sm_m[C][kRows], sm_l[C][kRows];
    __shared__ float c_m[kRows], c_l[kRows];
    __shared__ float s_f[C][kRows];
    __shared__ float s_fp[kMaxClusterSplits][kRows];
    __shared__ int64_t s_orow[kRows];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int split = blockIdx.y;
    const int nsplit = gridDim.y;
    const int bh = blockIdx.z;
    const int b = bh / p.Hkv;
    const int h = bh - b * p.Hkv;
    const bool early = p.prefetch != 0;
    const unsigned spin_limit = p.spin_limit;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 32);   // the owning producer's 32 lanes, each once its copies land
            mbar_init(&empty_bar[s], 1);   // the consuming warp's lane 0
        }
        if (CLUSTER && cluster_rank() == 0) mbar_init(&merge_bar, 1);
        mbar_init(&stall_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the cluster barrier phase opened here is closed before the first push (CTA 0's barrier is ready)
    if (CLUSTER) cluster_arrive_relaxed();
    __syncthreads();

    // Lengths, index lists and K/V rows may be read before the preceding kernel finishes when the caller
    // says they are ready (FX_LAUNCH_INPUTS_READY); everything else waits for it.
    if (!early) griddep_wait();
    // Split `split` of (b, h) takes one contiguous share of the index list and one contiguous share of
    // the tail, each in 16-key sub-tiles (only the last of a share may be partial): first nG gathered
    // sub-tiles (index entries ga .. gb-1), then the tail's (tokens ta .. tb-1).  The gathered share
    // depends only on the list length, so its copies go out while the length -- needed only for the
    // tail share and for the validity of each row -- is still being loaded.
    const int gper = (((p.kk + nsplit - 1) / nsplit + kSub - 1) / kSub) * kSub;
    const int ga = min(p.kk, split * gper);
    const int gb = min(p.kk, ga + gper);
    const int nG = (gb - ga + kSub - 1) / kSub;
    const int32_t* irow = p.idx != nullptr ? p.idx + (int64_t)bh * p.kk : nullptr;
    int len = __ldg(p.len + b);
    const bool bad_len = len < 0 || len > p.Tcap;
    len = len < 0 ? 0 : (len > p.Tcap ? p.Tcap : len);
    const int n_tail = max(0, len - p.tail_lo);
    const int tper = (((n_tail + nsplit - 1) / nsplit + kSub - 1) / kSub) * kSub;
    const int ta = p.tail_lo + min(n_tail, split * tper);
    const int tb = p.tail_lo + min(n_tail, split * tper + tper);
    auto n_local = [&]() { return nG + (tb - ta + kSub - 1) / kSub; };
    // token of row r of local sub-tile L whose K/V row is copied (-1: nothing to copy).  A gathered row
    // is copied when its index lies inside the cache's capacity; whether it counts (index < len) is
    // decided by the consumers, which also report rejected indices.
    auto copy_token = [&](int L, int r) {
        if (L < nG) {
            const int pos = ga + L * kSub + r;
            const int t = pos < gb ? __ldg(irow + pos) : -1;
            return (unsigned)t < (unsigned)p.Tcap ? t : -1;
        }
        const int t = ta + (L - nG) * kSub + r;
        return t < tb ? t : -1;
    };

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[n][e] = 0.f;

    if (warp >= C) {
        // ---------------- producers ----------------
        constexpr int kLA = kStreamMaxSlots / NP;   // own sub-tiles of index lookahead (one ring)
        const int pw = warp - C;
        const uint16_t* kb = p.k + (int64_t)b * p.sb + (int64_t)h * p.sh;
        const uint16_t* vb = p.v + (int64_t)b * p.sb + (int64_t)h * p.sh;
        const int r16 = lane & 15;   // the sub-tile row whose token this lane resolves
        const int c16 = lane & 15;   // the 16-byte chunk of a row this lane copies
        // own local sub-tiles L = pw + NP * i; index entries of the gathered ones, a ring ahead
        auto gathered_entry = [&](int i) {
            const int L = pw + NP * i;
            const int pos = ga + L * kSub + r16;
            return (L < nG && pos < gb) ? __ldg(irow + pos) : -1;
        };
        int tp[kLA];
#pragma unroll
        for (int q = 0; q < kLA; ++q) tp[q] = gathered_entry(q);
        int n_loc = -1;   // local sub-tiles, known once the length has arrived
        bool more = true;
        for (int ib = 0; more; ib += kLA) {
#pragma unroll
            for (int q = 0; q < kLA; ++q) {
                const int i = ib + q;
                const int L = pw + NP * i;
                if (L >= nG) {   // a tail sub-tile: the first one waits for the length
                    if (n_loc < 0) n_loc = n_local();
                    if (L >= n_loc) {
                        more = false;
                        break;
                    }
                }
                const int s = L % S;
                const int u = L / S;
                if (u > 0) mbar_wait_bounded(&empty_bar[s], (u - 1) & 1, p.err, spin_limit);
                unsigned char* stage = ring + (size_t)s * kSubBytes;
                if (L >= nG && p.tail_tma) {
                    // a contiguous tail sub-tile: four TMA boxes (K and V, columns 0-63 and 64-127); rows
                    // past this split's share are loaded but not used, rows past the capacity read as 0
                    if (lane == 0) {
                        const int t0 = ta + (L - nG) * kSub;
                        mbar_arrive_expect_tx_relaxed(&full_bar[s], (unsigned)kSubBytes);
                        const uint32_t st0 = smem_addr(stage);
                        tma_load_4d(st0, &tm_k, 0, t0, h, b, &full_bar[s]);
                        tma_load_4d(st0 + kHalfTile, &tm_k, 64, t0, h, b, &full_bar[s]);
                        tma_load_4d(st0 + 2 * kHalfTile, &tm_v, 0, t0, h, b, &full_bar[s]);
                        tma_load_4d(st0 + 3 * kHalfTile, &tm_v, 64, t0, h, b, &full_bar[s]);
                    } else {
                        mbar_arrive_relaxed(&full_bar[s]);
                    }
                } else {
                    int t;
                    if (L < nG) {
                        t = tp[q];
                        t = (unsigned)t < (unsigned)p.Tcap ? t : -1;
                    } else {
                        t = ta + (L - nG) * kSub + r16;
                        t = t < tb ? t : -1;
                    }
                    const bool ok = t >= 0;
                    const uint32_t vmask = __ballot_sync(kFull, ok) & 0xffffu;
                    const int64_t off = ok ? (int64_t)t * p.st : 0;
#pragma unroll
                    for (int u2 = 0; u2 < kSub / 2; ++u2) {
                        const int r = 2 * u2 + (lane >> 4);
                        const int64_t o_r = __shfl_sync(kFull, off, r);
                        const unsigned nb = ((vmask >> r) & 1u) ? 16u : 0u;
                        const uint32_t dk = smem_addr(stage + tile_off(r, c16));
                        cp_async16_fill(dk, kb + o_r + 8 * c16, nb);
                        cp_async16_fill(dk + 2 * kHalfTile, vb + o_r + 8 * c16, nb);
                    }
                    cp_async_mbar_arrive_noinc(&full_bar[s]);   // fires when this lane's copies have landed
                }
                tp[q] = gathered_entry(i + kLA);             // used kLA iterations later
            }
        }
        // Every copy of this split is issued: let the next call launch now, so that its ring fills during
        // this call's last round trip and merge rather than queueing ahead of this call's refills.  (This
        // CTA's own dependency wait comes first, as every dependent launch here requires.)
        griddep_wait();
        griddep_launch();
    } else {
        // ---------------- consumers ----------------
        // The query rows may be written by the preceding kernel, so they are read only after the wait;
        // an L2 prefetch is only a hint (L2 stays coherent with later writes) and shortens that read.
        if (tid < 2 * p.R) prefetch_l2(p.q + (((int64_t)b * p.Hq + h * p.G + (tid >> 1)) << 7) + 64 * (tid & 1));
        if (early) griddep_wait();
        const int g = lane >> 2;    // accumulator row: key g (and g + 8) of the sub-tile
        const int t4 = lane & 3;    // accumulator columns: query rows 2*t4, 2*t4 + 1
        // whether rows g and g + 8 of a sub-tile hold keys: the producer's copy test plus index < len;
        // the entries of this warp's first sub-tile are loaded now, later ones a sub-tile ahead
        const int n_loc = n_local();
        auto key_row = [&](int L, int r) { return L < n_loc ? copy_token(L, r) : -1; };
        int tok_a = key_row(warp, g);
        int tok_b = key_row(warp, g + 8);
        // the query rows of this (b, h) as one bf16 8-row tile (rows past R are zero)
        for (int e = tid; e < kRows * (kHeadDim / 8); e += 32 * C) {
            const int rr = e >> 4;
            const int c8 = e & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < p.R)
                v = *reinterpret_cast<const uint4*>(p.q + (((int64_t)b * p.Hq + h * p.G + rr) << 7) + c8 * 8);
            *reinterpret_cast<uint4*>(sQ + rr * kPitch + c8 * 16) = v;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(32 * C) : "memory");   // consumers only

        // padding rows (past R) see no key
        const bool live0 = 2 * t4 < p.R;
        const bool live1 = 2 * t4 + 1 < p.R;
        // B fragments of Q^T for the 8 k-steps of the 128-wide head
        uint32_t qf[8][2];
        {
            const int qrow = lane & 7;
            const int qcol = 8 * (lane >> 3);
#pragma unroll
            for (int kp = 0; kp < 4; ++kp)
                ldsm_x4(smem_addr(sQ + qrow * kPitch + (32 * kp + qcol) * 2), qf[2 * kp][0], qf[2 * kp][1],
                        qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
        }
        const int krow = (lane & 7) + 8 * ((lane >> 3) & 1);
        const int kcol = 8 * (lane >> 4);
        const int vrow = (lane & 7) + 8 * (lane >> 4);
        const int vcol = 8 * ((lane >> 3) & 1);
        for (int j = warp; j < n_loc; j += C) {
            const int s = j % S;
            const bool va = (unsigned)tok_a < (unsigned)len;
            const bool vb = (unsigned)tok_b < (unsigned)len;
            if (t4 == 0 && j < nG) {   // a listed index outside [0, len) is skipped and reported
                const int pos = ga + j * kSub + g;
                if ((pos < gb && !va) || (pos + 8 < gb && !vb)) flag(p.err, FX_DEVERR_INDEX);
            }
            tok_a = key_row(j + C, g);                   // the next sub-tile's, one iteration ahead
            tok_b = key_row(j + C, g + 8);
            mbar_wait_bounded(&full_bar[s], (j / S) & 1, p.err, spin_limit);
            const unsigned char* sk = ring + (size_t)s * kSubBytes;
            const unsigned char* sv = sk + 2 * kHalfTile;
            // S^T = K Q^T: 16 keys x 8 rows; two accumulators (even / odd k-steps) for independent chains
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ks += 2) {
                uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                ldsm_x4(smem_addr(sk + tile_off(krow, (16 * ks + kcol) >> 3)), a0, a1, a2, a3);
                ldsm_x4(smem_addr(sk + tile_off(krow, (16 * ks + 16 + kcol) >> 3)), c0, c1, c2, c3);
                mma_bf16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                mma_bf16(sb, c0, c1, c2, c3, qf[ks + 1][0], qf[ks + 1][1]);
            }
            // element e: key g + 8*(e >> 1) of the sub-tile, query row 2*t4 + (e & 1); base-2 logits
            float x[4];
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool ok = ((e >> 1) ? vb : va) && ((e & 1) ? live1 : live0);
                x[e] = ok ? (sa[e] + sb[e]) * p.qscale : -INFINITY;
                mx[e & 1] = fmaxf(mx[e & 1], x[e]);
            }
            float alpha[2], ms[2];
#pragma unroll
            for (int qc = 0; qc < 2; ++qc) {   // max over the 16 keys: the 8 lanes of this t4
                mx[qc] = fmaxf(mx[qc], __shfl_xor_sync(kFull, mx[qc], 4));
                mx[qc] = fmaxf(mx[qc], __shfl_xor_sync(kFull, mx[qc], 8));
                mx[qc] = fmaxf(mx[qc], __shfl_xor_sync(kFull, mx[qc], 16));
                const float mn = fmaxf(m_run[qc], mx[qc]);
                ms[qc] = (mn == -INFINITY) ? 0.f : mn;
                alpha[qc] = fast_exp2(m_run[qc] - ms[qc]);
                m_run[qc] = mn;
                l_run[qc] *= alpha[qc];
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                o[n][0] *= alpha[0];
                o[n][1] *= alpha[1];
                o[n][2] *= alpha[0];
                o[n][3] *= alpha[1];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[e] = fast_exp2(x[e] - ms[e & 1]);
                l_run[e & 1] += x[e];
            }
            // P^T as B fragments (the transpose of the (key g, rows 2t4..) layout), P = hi + lo in bf16
            uint32_t h01, l01, h23, l23;
            split_bf16(x[0], x[1], h01, l01);
            split_bf16(x[2], x[3], h23, l23);
            const uint32_t bh0 = movmatrix_t(h01), bh1 = movmatrix_t(h23);
            const uint32_t bl0 = movmatrix_t(l01), bl1 = movmatrix_t(l23);
            // O^T += V^T P^T: A fragments of V^T straight from the row-major V tile with ldmatrix.trans
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(smem_addr(sv + tile_off(vrow, (16 * mt + vcol) >> 3)), a0, a1, a2, a3);
                mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
                mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
            }
            __syncwarp();   // every lane has read the slot
            if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
    }
    // every thread has passed the dependency wait (the producer above) before anything is written
    __syncthreads();   // the ring is free: every copy landed and every slot was read
    if (bad_len && tid == 0) flag(p.err, FX_DEVERR_LEN);   // a length outside [0, capacity] was clamped
    // testing (fx_test_stall_wait): one bounded wait that runs out, exercising the give-up path
    if (p.test_stall != 0 && tid == 0) mbar_wait_bounded(&stall_bar, 0, p.err, p.test_stall);

    // ---- combine the consumer warps into this CTA's partial ---------------------------------------
    const int nr = min(kRows, p.R);
    float* sm_o = reinterpret_cast<float*>(ring);   // [C][8][kOPitch]
    if (warp < C) {
        const int g = lane >> 2;
        const int t4 = lane & 3;
#pragma unroll
        for (int qc = 0; qc < 2; ++qc) {   // sums over the 16 keys: the 8 lanes of this t4
            l_run[qc] += __shfl_xor_sync(kFull, l_run[qc], 4);
            l_run[qc] += __shfl_xor_sync(kFull, l_run[qc], 8);
            l_run[qc] += __shfl_xor_sync(kFull, l_run[qc], 16);
        }
#pragma unroll
        for (int qc = 0; qc < 2; ++qc) {
            const int r = 2 * t4 + qc;
            if (r < nr) {
                float* dst = sm_o + (warp * kRows + r) * kOPitch + g;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    dst[16 * mt] = o[mt][qc];
                    dst[16 * mt + 8] = o[mt][2 + qc];
                }
                if (g == 0) {
                    sm_m[warp][r] = m_run[qc];
                    sm_l[warp][r] = l_run[qc];
                }
            }
        }
    }
    __syncthreads();
    // per row, once: the CTA's maximum and sum, and each warp's weight 2^(m_w - M)
    if (tid < nr) {
        const int r = tid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C; ++w) M = fmaxf(M, sm_m[w][r]);
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < C; ++w) {
            const float f = fast_exp2(sm_m[w][r] - Ms);
            Ls = fmaf(sm_l[w][r], f, Ls);
            s_f[w][r] = f;
        }
        c_m[r] = M;
        c_l[r] = Ls;
        const int64_t orow = ((int64_t)b * p.Hq + h * p.G + r) << 7;
        s_orow[r] = orow;
    }
    __syncthreads();
    auto combined4 = [&](int r, int c) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < C; ++w) {
            const float f = s_f[w][r];
            const float4 v = *reinterpret_cast<const float4*>(sm_o + (w * kRows + r) * kOPitch + c);
            a.x = fmaf(v.x, f, a.x);
            a.y = fmaf(v.y, f, a.y);
            a.z = fmaf(v.z, f, a.z);
            a.w = fmaf(v.w, f, a.w);
        }
        return a;
    };

    int npeer = 0;
    if constexpr (CLUSTER) {
        // CTAs 1 .. nsplit-1 push their combined partial into CTA 0's receive area with asynchronous remote
        // stores that count their bytes on CTA 0's barrier, and exit; CTA 0 waits for them and merges.
        const unsigned me = cluster_rank();
        npeer = nsplit - 1;
        float* recv_m = s_recv + npeer * nr * kHeadDim;
        float* recv_l = recv_m + npeer * nr;
        cluster_wait_acquire();   // CTA 0's barrier is initialised
        if (me != 0) {
            const uint32_t rbar = cluster_map(&merge_bar, 0);
            const uint32_t dst = cluster_map(s_recv + (me - 1) * nr * kHeadDim, 0);
            for (int e = tid; e < nr * (kHeadDim / 4); e += blockDim.x)
                st_async_v4(dst + 16 * e, combined4(e >> 5, 4 * (e & 31)), rbar);
            if (tid < nr) {
                st_async_f32(cluster_map(recv_m + (me - 1) * nr + tid, 0), c_m[tid], rbar);
                st_async_f32(cluster_map(recv_l + (me - 1) * nr + tid, 0), c_l[tid], rbar);
            }
            return;
        }
        if (tid == 0) mbar_arrive_expect_tx(&merge_bar, (unsigned)(npeer * nr * (kHeadDim + 2) * 4));
        unsigned spins = 0;
        while (!mbar_try_wait_cluster(&merge_bar, 0)) {
            if (++spins >= spin_limit) {
                if (tid == 0) flag(p.err, FX_DEVERR_TIMEOUT);
                break;
            }
        }
        // per row, once: the weights of this CTA's warps and of each peer with 1 / L folded in
        if (tid < nr) {
            const int r = tid;
            float M = c_m[r];
            for (int q = 0; q < npeer; ++q) M = fmaxf(M, recv_m[q * nr + r]);
            const float Ms = (M == -INFINITY) ? 0.f : M;
            const float a0 = fast_exp2(c_m[r] - Ms);
            float Ls = c_l[r] * a0;
            for (int q = 0; q < npeer; ++q) {
                const float aq = fast_exp2(recv_m[q * nr + r] - Ms);
                Ls = fmaf(recv_l[q * nr + r], aq, Ls);
                s_fp[q][r] = aq;
            }
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
            for (int w = 0; w < C; ++w) s_f[w][r] *= a0 * inv;
            for (int q = 0; q < npeer; ++q) s_fp[q][r] *= inv;
        }
    } else {
        if (tid < nr) {
            const float inv = c_l[tid] > 0.f ? 1.f / c_l[tid] : 0.f;
#pragma unroll
            for (int w = 0; w < C; ++w) s_f[w][tid] *= inv;
        }
    }
    __syncthreads();
    for (int e = tid; e < nr * (kHeadDim / 4); e += blockDim.x) {
        const int r = e >> 5;
        const int c = 4 * (e & 31);
        float4 a = combined4(r, c);
        for (int q = 0; q < npeer; ++q) {
            const float f = s_fp[q][r];
            const float4 v = *reinterpret_cast<const float4*>(s_recv + (q * nr + r) * kHeadDim + c);
            a.x = fmaf(v.x, f, a.x);
            a.y = fmaf(v.y, f, a.y);
            a.z = fmaf(v.z, f, a.z);
            a.w = fmaf(v.w, f, a.w);
        }
        *reinterpret_cast<float4*>(p.out + s_orow[r] + c) = a;
    }
}

template <int C, int NP, bool CLUSTER>
cudaError_t launch_stream_one(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, size_t smem, bool pdl,
                              cudaStream_t s)
{
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = stream_decode_kernel<C, NP, CLUSTER>;
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmemMax);
        if (e != cudaSuccess) return e;
        // the whole unified L1 / shared array as shared memory, so two CTAs fit one SM
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        if (CLUSTER) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        configured = dev;
    }
    dim3 grid(1, p.nsplit, p.B * p.Hkv);
    return launch_kernel(kern, grid, dim3(32 * (C + NP)), smem, s, pdl, CLUSTER ? (unsigned)p.nsplit : 0u, p, tk, tv);
}

}  // namespace

size_t stream_decode_smem_bytes(int slots, int nsplit, int R)
{
    const int nr = R < kRows ? R : kRows;
    const size_t recv = (size_t)(nsplit - 1) * nr * (kHeadDim + 2) * sizeof(float);
    return 1024 + (size_t)slots * kSubBytes + (size_t)kRows * kPitch + ((recv + 15) / 16) * 16;
}

cudaError_t launch_stream_decode(const AttnParams& p, const CUtensorMap* tk, const CUtensorMap* tv, bool pdl,
                                 cudaStream_t s)
{
    if (p.R > kRows || p.Mq != 1 || p.stages < kStreamProducers || p.stages > kStreamMaxSlots ||
        p.stages % kStreamProducers != 0 || p.nsplit < 1 || p.nsplit > kMaxClusterSplits)
        return cudaErrorInvalidValue;
    const size_t smem = stream_decode_smem_bytes(p.stages, p.nsplit, p.R);
    if (smem > kStreamSmemMax) return cudaErrorInvalidValue;
    if (p.tail_tma && (tk == nullptr || tv == nullptr)) return cudaErrorInvalidValue;
    static const CUtensorMap unused = {};
    const CUtensorMap& k = p.tail_tma ? *tk : unused;
    const CUtensorMap& v = p.tail_tma ? *tv : unused;
    if (p.nsplit == 1) return launch_stream_one<kStreamConsumers, kStreamProducers, false>(p, k, v, smem, pdl, s);
    return launch_stream_one<kStreamConsumers, kStreamProducers, true>(p, k, v, smem, pdl, s);
}

}  // namespace fx
