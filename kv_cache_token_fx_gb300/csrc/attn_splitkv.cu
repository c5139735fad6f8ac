// Split-KV decode / verify attention for sm_103a.
//
// One CTA (4 warps) = (group of NR = 8, 16 or 32 query rows of one KV head, one split of that head's
// key sequence, one (b, KV head)).  Each warp owns a contiguous range of whole 16-key sub-tiles of the
// split (a fixed quarter of it; in the prefix mode a quarter of the keys the row actually has) and
// walks it on its own:
//   * Data movement: the warp stages its sub-tiles (16 K rows + 16 V rows of 256 bytes; contiguous
//     rows for the focal mode, gathered rows for the sparse/prefix modes) into a private ring of
//     2 or 3 buffers (attn_stages) with 16-byte cp.async, each warp instruction moving two whole
//     rows, one commit group per sub-tile, so no CTA-wide barrier is needed in the loop.  Lane l
//     resolves the token of row l & 15 (one index load per lane); the copies take the row addresses
//     by warp shuffle and a ballot records which rows are valid.  Within a row the 16-byte chunk index
//     is XORed with (row % 8), so the 8-row ldmatrix reads hit 8 different bank groups without
//     padding; invalid rows are zero-filled.  (Per-row cp.async.bulk TMA copies were measured slower
//     here: 256-byte requests keep the TMA engine, not HBM, busy.)
//   * Math: mma.sync m16n8k16 (bf16 in, fp32 accumulate), online softmax on the accumulator
//     fragments in base-2 units, P split into bf16 hi + lo parts (two MMAs) so that the
//     probabilities keep ~16 bits.  With NR = 8 the keys are the M side (S^T = K Q^T, O^T = V^T P^T,
//     P^T moved into the B operand with movmatrix.trans): half the MMAs of the NR = 16 layout, where
//     the query rows are the M side (S = Q K^T, O = P V).  NR = 32 (scoring-only focal calls) keeps
//     the keys on M with four query n-tiles sharing each K fragment, and has no P V.
// The warps' partials are combined with per-row weights computed once.  Partial (max, sum,
// unnormalised output) triples per split are merged inside a thread-block cluster -- all splits of
// one (b, h, row group) form one cluster; either the others push their partials into CTA 0 with
// st.async (completing on CTA 0's mbarrier) and exit, or every CTA reads all partials from
// distributed shared memory -- or, for the focal call and for very long rows, through the workspace
// (the focal call's combine kernel also forms the per-token importance from the logits this kernel
// stores).  A verify call whose dense prefix ran on the tensor cores folds that partial in here.
//
// Attention and importance follow FastOCR (Methodology: Focal-Guided Pruning): focal layers attend
// over the full cache, the rest over the selected set; FastKV (2.A) for the causal query window;
// HPD-Parsing (parts 2 and 3) for the shared prefix + private suffix + causal draft sequence.
#include <cuda_bf16.h>
#include <math.h>

#include "attn_ptx.cuh"
#include "fx_internal.h"

namespace fx {
namespace {

// ---- key sequences --------------------------------------------------------------------------------
// Where the rows of one (b, h) key sequence live: sequence position -> K row and V row.
template <int MODE>
struct KeySource {
    const uint16_t* kb;   // main cache / prefix base for this (b, h)
    const uint16_t* vb;
    int64_t st;
    const int32_t* irow;  // gathered positions of this (b, h) (sparse idx / prefix idx), or null
    int kk;               // number of gathered positions
    int lim_tok;          // exclusive bound of a gathered position (len for sparse, P for prefix)
    int tail_lo;          // sparse: first tail token
    int np, L;            // prefix: prefix rows, suffix rows
    const uint16_t* suf_k;
    const uint16_t* suf_v;
    int64_t suf_st;
    const uint16_t* dr_k;
    const uint16_t* dr_v;
    int64_t dr_si;
    unsigned* err;

    // Token of sequence position pos: an index-row load for the gathered part (only for pos < kk, so
    // always inside the row), the position itself otherwise.  Nothing is checked here.
    __device__ __forceinline__ int token(int pos) const
    {
        if (MODE == kModeSparse) return pos < kk ? __ldg(irow + pos) : tail_lo + (pos - kk);
        if (MODE == kModePrefix) return (irow != nullptr && pos < kk) ? __ldg(irow + pos) : pos;
        return pos;
    }

    // K and V rows of position pos whose token is t; false when they must not be read (a rejected
    // index, which is also reported in the device error word).
    __device__ __forceinline__ bool row(int pos, int t, const uint16_t*& kp, const uint16_t*& vp) const
    {
        if (MODE == kModeFocal) {
            kp = kb + (int64_t)t * st;
            vp = vb + (int64_t)t * st;
            return true;
        }
        if (MODE == kModeSparse || pos < np) {
            const bool gathered = MODE == kModeSparse ? pos < kk : irow != nullptr;
            if (gathered && (t < 0 || t >= lim_tok)) {
                atomicOr(err, FX_DEVERR_INDEX);
                return false;
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

// ---- the kernel -----------------------------------------------------------------------------------
// Output value from the split-merged (M, and Ls, O relative to Ms).  A partial over other keys of the
// row computed by another kernel (ext: the dense shared prefix of the verify call; me = -inf when
// absent) is folded in first.
__device__ __forceinline__ float finish_row(float me, float le, float oe, float M, float Ms, float Ls, float O)
{
    if (me != -INFINITY) {
        const float mn = fmaxf(M, me);
        const float a = M == -INFINITY ? 0.f : fast_exp2(Ms - mn);
        const float e = fast_exp2(me - mn);
        Ls = fmaf(Ls, a, le * e);
        O = fmaf(O, a, oe * e);
    }
    return Ls > 0.f ? O / Ls : 0.f;
}

// How the splits of one (b, h, row group) are merged.
enum Merge {
    kMergeWorkspace = 0,   // partials through the workspace; the last-arriving CTA merges
    kMergePull = 1,        // one cluster; every CTA reads all partials from distributed shared memory
    kMergePush = 2,        // one cluster; the others push their partials into CTA 0, which merges alone
};

template <int MODE, int MERGE, int NR>
__global__ void __launch_bounds__(kThreads) attn_tile_kernel(const AttnParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sQ = smem + 128;                                      // [16][kPitch] bf16
    constexpr int WS = attn_stages(MODE);                               // sub-tiles in flight per warp
    constexpr int kWarpBytes = WS * kSubBytes;                          // one warp's ring of sub-tile buffers
    unsigned char* sKV = sQ + attn_q_rows(NR) * kPitch;                  // [kWarps][WS][K, V]
    __shared__ uint32_t s_vmask[kWarps][WS];   // valid-row bits of each staged sub-tile

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int g = lane >> 2;      // accumulator row within the 16-row tile (and row + 8)
    const int t4 = lane & 3;      // accumulator column pair
    const int rg = blockIdx.x;
    const int split = blockIdx.y;
    const int bh = blockIdx.z;
    const int b = bh / p.Hkv;
    const int h = bh - b * p.Hkv;
    const int r0 = rg * NR;

    // ---- stage A: what depends only on the caller's lengths, indices and K/V rows.  With
    // FX_LAUNCH_INPUTS_READY it runs before the preceding kernel on the stream has finished, so the
    // first tiles are already in flight when that kernel ends.
    const bool early = p.prefetch != 0;
    // kMergePush: CTA 0's barrier for the pushed partials, initialised before anything else; the cluster
    // barrier phase opened here (closed before the first push) makes the initialisation visible.
    __shared__ __align__(8) uint64_t s_merge_bar;
    if constexpr (MERGE == kMergePush) {
        if (tid == 0 && cluster_rank() == 0) mbar_init_for_cluster(&s_merge_bar, 1);
        cluster_arrive_relaxed();
    }
    if (!early) griddep_wait();

    // key sequence of this (b, h)
    KeySource<MODE> src;
    int n_keys;
    src.kb = p.k + (int64_t)b * p.sb + (int64_t)h * p.sh;
    src.vb = p.v + (int64_t)b * p.sb + (int64_t)h * p.sh;
    src.st = p.st;
    src.kk = p.kk;
    src.tail_lo = p.tail_lo;
    src.irow = p.idx != nullptr ? p.idx + (int64_t)bh * p.kk : nullptr;
    src.err = p.err;
    src.np = 0;
    src.L = 0;
    src.lim_tok = p.P;
    // this warp's contiguous share of the split (the host makes split_len a multiple of kWarps * kSub),
    // and the index loads of its first sub-tiles, issued before the length is known
    const int s0 = split * p.split_len;
    int wl = p.split_len / kWarps;
    int ws = s0 + warp * wl;
    int tpre[WS];
#pragma unroll
    for (int j = 0; j < WS; ++j) tpre[j] = MODE == kModePrefix ? 0 : src.token(ws + j * kSub + (lane & 15));

    if (MODE == kModeFocal || MODE == kModeSparse) {
        int l = p.len[b];
        if (l < 0 || l > p.Tcap) {
            if (tid == 0) flag(p.err, FX_DEVERR_LEN);
            l = l < 0 ? 0 : p.Tcap;
        }
        n_keys = (MODE == kModeFocal) ? l : p.kk + max(0, l - p.tail_lo);
        src.lim_tok = l;
    } else {
        // the prefix rows this branch sees: all P, or its fork position
        int pb = p.P;
        if (p.pre_len != nullptr) {
            pb = p.pre_len[b];
            if (pb < 0 || pb > p.P) {
                if (tid == 0) flag(p.err, FX_DEVERR_LEN);
                pb = pb < 0 ? 0 : p.P;
            }
        }
        src.np = p.idx ? p.kk : pb;
        src.lim_tok = pb;
        const int o0 = p.suf_off[b];
        const int64_t o1 = p.suf_len != nullptr ? (int64_t)o0 + p.suf_len[b] : (int64_t)p.suf_off[b + 1];
        int L = 0;
        if (o0 < 0 || o1 < o0 || o1 > p.suf_rows) {
            if (tid == 0) flag(p.err, FX_DEVERR_OFFSETS);
        } else {
            L = (int)(o1 - o0);
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
    const int s1 = min(n_keys, s0 + p.split_len);
    if (MODE == kModePrefix) {
        // verify rows differ in length (private suffixes): the warps share this split's actual keys, so
        // a short row does not leave most of them idle
        const int share = (max(0, s1 - s0) + kWarps * kSub - 1) / (kWarps * kSub) * kSub;
        wl = share;
        ws = s0 + warp * share;
#pragma unroll
        for (int j = 0; j < WS; ++j) tpre[j] = src.token(ws + j * kSub + (lane & 15));
    }
    const int we = min(s1, ws + wl);
    const int nsub = we > ws ? (we - ws + kSub - 1) / kSub : 0;

    // Each warp stages its own sub-tiles (16 K rows + 16 V rows) with 16-byte cp.async operations --
    // every warp instruction moves two whole rows -- into its private ring of WS buffers.  One
    // commit group per sub-tile (empty past the end), so "all but WS-1 groups done" always
    // means "the oldest sub-tile has landed".  No CTA-wide barrier is needed inside the loop.
    unsigned char* wbuf = sKV + (size_t)warp * kWarpBytes;
    // a focal call that only scores (no output rows) needs no V rows and no P V products
    const bool need_v = NR != 32 && !(MODE == kModeFocal && p.no_v);
    auto issue = [&](int j, int mytok) {
        if (j < nsub) {
            const int c16 = lane & 15;
            unsigned char* stage = wbuf + (size_t)(j % WS) * kSubBytes;
            // lane l resolves the token row of key (l & 15) of the sub-tile (one index load per lane);
            // the copies then take each row's address from the lane that resolved it
            const int mypos = ws + j * kSub + (lane & 15);
            const uint16_t* mk = src.kb;
            const uint16_t* mv = src.vb;
            const bool mok = mypos < we && src.row(mypos, mytok, mk, mv);
            const uint32_t vmask = __ballot_sync(kFull, mok) & 0xffffu;
            const int64_t mko = mk - src.kb;
            const int64_t mvo = mv - src.vb;
#pragma unroll
            for (int u = 0; u < kSub / 2; ++u) {
                const int r = 2 * u + (lane >> 4);
                const uint16_t* kp = src.kb + __shfl_sync(kFull, mko, r);
                const uint16_t* vp = src.vb + (MODE == kModePrefix ? __shfl_sync(kFull, mvo, r)
                                                                   : __shfl_sync(kFull, mko, r));
                unsigned char* dk = stage + kv_off(r, c16);
                unsigned char* dv = dk + kSub * kKvPitch;
                if ((vmask >> r) & 1u) {
                    cp_async16(smem_addr(dk), kp + 8 * c16);
                    if (need_v) cp_async16(smem_addr(dv), vp + 8 * c16);
                } else {
                    *reinterpret_cast<uint4*>(dk) = make_uint4(0u, 0u, 0u, 0u);
                    if (need_v) *reinterpret_cast<uint4*>(dv) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (lane == 0) s_vmask[warp][j % WS] = vmask;
        }
        cp_async_commit();
    };

#pragma unroll
    for (int j = 0; j < WS; ++j) issue(j, tpre[j]);

    // The query rows may be written by the preceding kernel, so they are read only after the wait
    // below; a prefetch into L2 is only a hint (L2 stays coherent with later writes) and shortens that
    // read when the rows were not in L2 yet.  Two 128-byte lines per row.
    if (tid < 2 * NR && r0 + (tid >> 1) < p.R) {
        const int row = r0 + (tid >> 1);
        const int gi = row / p.Mq;
        const int i = row - gi * p.Mq;
        prefetch_l2(p.q + ((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + 64 * (tid & 1));
    }

    // ---- stage B: after the preceding kernel -- the query rows, then everything that writes ------
    if (early) griddep_wait();
    griddep_launch();

    // the query rows of this group as one bf16 NR-row tile (rows past R are zero)
    for (int e = tid; e < NR * (kHeadDim / 8); e += kThreads) {
        const int rr = e >> 4;
        const int c8 = e & 15;
        const int row = r0 + rr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < p.R) {
            const int gi = row / p.Mq;
            const int i = row - gi * p.Mq;
            v = *reinterpret_cast<const uint4*>(p.q + ((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + c8 * 8);
        }
        *reinterpret_cast<uint4*>(sQ + rr * kPitch + c8 * 16) = v;
    }
    __syncthreads();

    // Visibility limit of one query row: the last key position it may see.
    auto row_limit = [&](int row) {
        const int i = row - (row / p.Mq) * p.Mq;
        if (row >= p.R) return -1;   // padding row: sees nothing
        if (MODE == kModeFocal) return p.q_pos0 >= 0 ? p.q_pos0 + i : 0x7fffffff;
        if (MODE == kModePrefix) return src.np + src.L + i;   // draft row j is visible iff j <= i
        return 0x7fffffff;
    };

    // Two layouts of the per-warp math (both mma.sync m16n8k16, bf16 in, fp32 accumulate):
    //   NR == 16 (wide): the query rows are the M side.  S = Q K^T is a 16-row x 16-key tile (2 n-tiles),
    //     O = P V accumulates 16 rows x 128 dims.  48 MMAs per 16 keys.
    //   NR == 8 (narrow, at most 8 query rows): the keys are the M side.  S^T = K Q^T is 16 keys x 8 rows
    //     (one tile per k-step), O^T = V^T P^T accumulates 128 dims x 8 rows; P^T reaches the B operand
    //     through movmatrix.trans.  24 MMAs per 16 keys -- half the tensor work when few rows exist.
    //   NR == 32 (scores only: no output rows): keys on M as for 8 rows, with 4 n-tiles of 8 query rows
    //     sharing every K fragment, so K is read once for up to 32 rows.  32 MMAs per 16 keys, no P V.
    constexpr int kNT = NR == 32 ? 4 : 1;                       // query n-tiles of the narrow layouts
    constexpr int kOT = NR == 8 ? 8 : (NR == 32 ? 1 : 16);      // accumulator tiles of O (wide) / O^T (narrow)
    constexpr int kQF = NR == 16 ? 4 : 2 * kNT;                 // registers of one k-step's Q fragment
    int lim[2 * kNT];
    uint32_t qf[8][kQF];
    if constexpr (NR == 32) {
        // n-tile nt, column qc: query row 8*nt + 2*t4 + qc
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            lim[2 * nt] = row_limit(r0 + 8 * nt + 2 * t4);
            lim[2 * nt + 1] = row_limit(r0 + 8 * nt + 2 * t4 + 1);
        }
        const int qrow = lane & 7;
        const int qcol = 8 * (lane >> 3);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int kp = 0; kp < 4; ++kp)
                ldsm_x4(smem_addr(sQ + (8 * nt + qrow) * kPitch + (32 * kp + qcol) * 2), qf[2 * kp][2 * nt],
                        qf[2 * kp][2 * nt + 1], qf[2 * kp + 1][2 * nt], qf[2 * kp + 1][2 * nt + 1]);
    } else if constexpr (NR == 8) {
        // this thread's accumulator columns are query rows 2*t4 and 2*t4 + 1
        lim[0] = row_limit(r0 + 2 * t4);
        lim[1] = row_limit(r0 + 2 * t4 + 1);
        // B fragments of Q^T: matrices (rows 0-7, dims 32kp + 0/8/16/24 .. +7)
        const int qrow = lane & 7;
        const int qcol = 8 * (lane >> 3);
#pragma unroll
        for (int kp = 0; kp < 4; ++kp)
            ldsm_x4(smem_addr(sQ + qrow * kPitch + (32 * kp + qcol) * 2), qf[2 * kp][0], qf[2 * kp][1],
                    qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
    } else {
        // this thread's accumulator rows are g and g + 8
        lim[0] = row_limit(r0 + g);
        lim[1] = row_limit(r0 + g + 8);
        // A fragments of Q for the 8 k-steps of the 128-wide head
        const int qrow = (lane & 7) + 8 * ((lane >> 3) & 1);
        const int qcol = 8 * (lane >> 4);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            ldsm_x4(smem_addr(sQ + qrow * kPitch + (16 * ks + qcol) * 2), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }

    float o[kOT][4];
#pragma unroll
    for (int n = 0; n < kOT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
    float m_run[2 * kNT], l_run[2 * kNT];      // per accumulator row (wide) / query column (narrow)
#pragma unroll
    for (int i = 0; i < 2 * kNT; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
    }
    for (int j = 0; j < nsub; ++j) {
        const int base = ws + j * kSub;   // first key of this sub-tile
        const int tnext = src.token(base + WS * kSub + (lane & 15));   // for the refill below
        cp_async_wait_stages<WS>();
        __syncwarp();
        const unsigned char* sk = wbuf + (size_t)(j % WS) * kSubBytes;
        const unsigned char* sv = sk + kSub * kKvPitch;
        const uint32_t vmask = s_vmask[warp][j % WS];

        if constexpr (NR == 32) {
            // S^T = K Q^T for 4 n-tiles of 8 query rows; each K fragment serves all four
            float acc[kNT][4];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
            {
                const int krow = (lane & 7) + 8 * ((lane >> 3) & 1);
                const int kcol = 8 * (lane >> 4);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(smem_addr(sk + kv_off(krow, (16 * ks + kcol) >> 3)), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt) mma_bf16(acc[nt], a0, a1, a2, a3, qf[ks][2 * nt], qf[ks][2 * nt + 1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                // element e: key g + 8*(e >> 1) of the sub-tile, query row 8*nt + 2*t4 + (e & 1)
                float x[4];
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kr = g + 8 * (e >> 1);
                    const int qc = e & 1;
                    const bool ok = ((vmask >> kr) & 1u) && base + kr <= lim[2 * nt + qc];
                    x[e] = ok ? acc[nt][e] * p.qscale : -INFINITY;
                    mx[qc] = fmaxf(mx[qc], x[e]);
                }
                if (p.logits != nullptr) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = r0 + 8 * nt + 2 * t4 + (e & 1);
                        const int pos = base + g + 8 * (e >> 1);
                        if (row < p.R && pos < we) p.logits[(int64_t)(bh * p.R + row) * p.Tcap + pos] = x[e];
                    }
                }
#pragma unroll
                for (int qc = 0; qc < 2; ++qc) {   // max over the 16 keys: the 8 lanes of this t4
                    mx[qc] = fmaxf(mx[qc], __shfl_xor_sync(kFull, mx[qc], 4));
                    mx[qc] = fmaxf(mx[qc], __shfl_xor_sync(kFull, mx[qc], 8));
                    mx[qc] = fmaxf(mx[qc], __shfl_xor_sync(kFull, mx[qc], 16));
                    const float mn = fmaxf(m_run[2 * nt + qc], mx[qc]);
                    const float ms = (mn == -INFINITY) ? 0.f : mn;
                    l_run[2 * nt + qc] *= fast_exp2(m_run[2 * nt + qc] - ms);
                    m_run[2 * nt + qc] = mn;
#pragma unroll
                    for (int e = qc; e < 4; e += 2) l_run[2 * nt + qc] += fast_exp2(x[e] - ms);
                }
            }
        } else if constexpr (NR == 8) {
            // S^T = K Q^T: 16 keys x 8 rows; two accumulators (even / odd k-steps) for independent chains
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const int krow = (lane & 7) + 8 * ((lane >> 3) & 1);
                const int kcol = 8 * (lane >> 4);
#pragma unroll
                for (int ks = 0; ks < 8; ks += 2) {
                    uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                    ldsm_x4(smem_addr(sk + kv_off(krow, (16 * ks + kcol) >> 3)), a0, a1, a2, a3);
                    ldsm_x4(smem_addr(sk + kv_off(krow, (16 * ks + 16 + kcol) >> 3)), c0, c1, c2, c3);
                    mma_bf16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                    mma_bf16(sb, c0, c1, c2, c3, qf[ks + 1][0], qf[ks + 1][1]);
                }
            }
            // element e: key g + 8*(e >> 1) of the sub-tile, query column 2*t4 + (e & 1)
            float x[4];
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kr = g + 8 * (e >> 1);
                const int qc = e & 1;
                const bool ok = ((vmask >> kr) & 1u) && base + kr <= lim[qc];
                x[e] = ok ? (sa[e] + sb[e]) * p.qscale : -INFINITY;
                mx[qc] = fmaxf(mx[qc], x[e]);
            }
            if (MODE == kModeFocal && p.logits != nullptr) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = r0 + 2 * t4 + (e & 1);
                    const int pos = base + g + 8 * (e >> 1);
                    if (row < p.R && pos < we) p.logits[(int64_t)(bh * p.R + row) * p.Tcap + pos] = x[e];
                }
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
            for (int n = 0; n < kOT; ++n) {
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
            // P^T as B fragments: (keys 2t4.., row g) = the transpose of the (key g, rows 2t4..) layout;
            // P = hi + lo in bf16
            if (need_v) {
                uint32_t h01, l01, h23, l23;
                split_bf16(x[0], x[1], h01, l01);
                split_bf16(x[2], x[3], h23, l23);
                const uint32_t bh0 = movmatrix_t(h01), bh1 = movmatrix_t(h23);
                const uint32_t bl0 = movmatrix_t(l01), bl1 = movmatrix_t(l23);
                // O^T += V^T P^T: A fragments of V^T straight from the row-major V tile with ldmatrix.trans
                const int vrow = (lane & 7) + 8 * (lane >> 4);
                const int vcol = 8 * ((lane >> 3) & 1);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(smem_addr(sv + kv_off(vrow, (16 * mt + vcol) >> 3)), a0, a1, a2, a3);
                    mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
                    mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
                }
            }
        } else {
            // S = Q K^T for this warp's 16 keys (2 n-tiles of 8 keys)
            float s[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
                const int krow = 8 * nt + (lane & 7);
                const int kcol = 8 * (lane >> 3);   // matrices: dims +0, +8, +16, +24 of a 32-dim slice
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {     // pairs of k-steps
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_addr(sk + kv_off(krow, (32 * kp + kcol) >> 3)), b0, b1, b2, b3);
                    mma_bf16(s[nt], qf[2 * kp][0], qf[2 * kp][1], qf[2 * kp][2], qf[2 * kp][3], b0, b1);
                    mma_bf16(s[nt], qf[2 * kp + 1][0], qf[2 * kp + 1][1], qf[2 * kp + 1][2], qf[2 * kp + 1][3], b2, b3);
                }
            }

            // scale to base 2, mask, store logits (focal), online softmax
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int hr = e >> 1;
                    const int pos = base + 8 * nt + 2 * t4 + (e & 1);
                    const bool ok = ((vmask >> (pos - base)) & 1u) && pos <= lim[hr];
                    const float x = ok ? s[nt][e] * p.qscale : -INFINITY;
                    s[nt][e] = x;
                    mx[hr] = fmaxf(mx[hr], x);
                }
            }
            if (MODE == kModeFocal && p.logits != nullptr) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int row = r0 + g + 8 * hr;
                    if (row < p.R) {
                        float* lrow = p.logits + (int64_t)(bh * p.R + row) * p.Tcap;
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const int pos = base + 8 * nt + 2 * t4;
                            if (pos < we) lrow[pos] = s[nt][2 * hr];
                            if (pos + 1 < we) lrow[pos + 1] = s[nt][2 * hr + 1];
                        }
                    }
                }
            }
            // the running maximum moves only when the sub-tile's maximum exceeds it by more than
            // kMaxSlack, so O is rescaled a few times per row instead of every sub-tile (P <= 2^kMaxSlack)
            float alpha[2], ms[2];
            bool grow_any = false;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(kFull, mx[hr], 1));
                mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(kFull, mx[hr], 2));
                const bool grow = mx[hr] > m_run[hr] + kMaxSlack;   // also: first keys of the row
                const float mn = grow ? mx[hr] : m_run[hr];
                ms[hr] = (mn == -INFINITY) ? 0.f : mn;
                alpha[hr] = grow ? fast_exp2(m_run[hr] - ms[hr]) : 1.f;
                m_run[hr] = mn;
                l_run[hr] *= alpha[hr];
                grow_any |= grow;
            }
            if (__any_sync(kFull, grow_any)) {
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    o[n][0] *= alpha[0];
                    o[n][1] *= alpha[0];
                    o[n][2] *= alpha[1];
                    o[n][3] *= alpha[1];
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pe = fast_exp2(s[nt][e] - ms[e >> 1]);
                    s[nt][e] = pe;
                    l_run[e >> 1] += pe;
                }
            }

            // O += P V over this warp's 16 keys (one k-step); P = hi + lo in bf16
            if (need_v) {
                uint32_t ph[4], pl[4];
                split_bf16(s[0][0], s[0][1], ph[0], pl[0]);
                split_bf16(s[0][2], s[0][3], ph[1], pl[1]);
                split_bf16(s[1][0], s[1][1], ph[2], pl[2]);
                split_bf16(s[1][2], s[1][3], ph[3], pl[3]);
                const int vrow = (lane & 7) + 8 * ((lane >> 3) & 1);
                const int vcol = 8 * (lane >> 4);
#pragma unroll
                for (int np2 = 0; np2 < 8; ++np2) {   // pairs of 8-dim n-tiles
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_addr(sv + kv_off(vrow, (16 * np2 + vcol) >> 3)), b0, b1, b2, b3);
                    mma_bf16(o[2 * np2], ph[0], ph[1], ph[2], ph[3], b0, b1);
                    mma_bf16(o[2 * np2], pl[0], pl[1], pl[2], pl[3], b0, b1);
                    mma_bf16(o[2 * np2 + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
                    mma_bf16(o[2 * np2 + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
                }
            }
        }

        __syncwarp();      // every lane is done with this buffer before it is refilled
        issue(j + WS, tnext);
    }
    // the external partial of these rows (column tid of each; kThreads == kHeadDim), loaded now so its
    // latency overlaps the combine below
    static_assert(kThreads == kHeadDim, "one output column per thread");
    constexpr int kExtRows = NR == 32 ? 1 : NR;
    float ext_oc[kExtRows];
    __shared__ float s_ext_m[kMaxRowsPerCta];
    __shared__ float s_ext_l[kMaxRowsPerCta];
#pragma unroll
    for (int r = 0; r < kExtRows; ++r) ext_oc[r] = 0.f;
    if (NR != 32 && p.ext_m != nullptr) {
        const int64_t er0 = ((int64_t)h * p.B + b) * p.R + r0;
#pragma unroll
        for (int r = 0; r < kExtRows; ++r)
            if (r0 + r < p.R) ext_oc[r] = __ldcg(p.ext_o + (er0 + r) * kHeadDim + tid);
        if (tid < NR && r0 + tid < p.R) {
            s_ext_m[tid] = __ldcg(p.ext_m + er0 + tid);
            s_ext_l[tid] = __ldcg(p.ext_l + er0 + tid);
        }
    } else if (tid < kMaxRowsPerCta) {
        s_ext_m[tid] = -INFINITY;
        s_ext_l[tid] = 0.f;
    }
    cp_async_wait_all_groups();
    __syncthreads();       // all warps are done with their buffers (reused below)

    // ---- combine the warps into this CTA's partial (the stage buffers are free now) -------------
    const int nr = min(NR, p.R - r0);   // rows of this group that exist
    __shared__ float sm_m[kWarps][kMaxRowsPerCta];
    __shared__ float sm_l[kWarps][kMaxRowsPerCta];
    // [kWarps][16][kOPitch]: rows padded by 8 floats, so the row-strided fragment stores of the
    // 16-row path spread over all banks
    constexpr int kOPitch = kHeadDim + 8;
    float* sm_o = reinterpret_cast<float*>(sKV);
    if constexpr (NR == 32) {
#pragma unroll
        for (int i = 0; i < 2 * kNT; ++i) {   // sums over the 16 keys: the 8 lanes of this t4
            l_run[i] += __shfl_xor_sync(kFull, l_run[i], 4);
            l_run[i] += __shfl_xor_sync(kFull, l_run[i], 8);
            l_run[i] += __shfl_xor_sync(kFull, l_run[i], 16);
        }
        if (g == 0) {
#pragma unroll
            for (int i = 0; i < 2 * kNT; ++i) {
                const int r = 8 * (i >> 1) + 2 * t4 + (i & 1);
                if (r < nr) {
                    sm_m[warp][r] = m_run[i];
                    sm_l[warp][r] = l_run[i];
                }
            }
        }
    } else if constexpr (NR == 8) {
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
                float* dst = sm_o + (warp * kRowsPerCta + r) * kOPitch + g;
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
    } else {
        // row sums over the quad
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            l_run[hr] += __shfl_xor_sync(kFull, l_run[hr], 1);
            l_run[hr] += __shfl_xor_sync(kFull, l_run[hr], 2);
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {   // only the rows that exist
            const int c = 8 * n + 2 * t4;
            if (g < nr) *reinterpret_cast<float2*>(sm_o + (warp * kRowsPerCta + g) * kOPitch + c) = make_float2(o[n][0], o[n][1]);
            if (g + 8 < nr)
                *reinterpret_cast<float2*>(sm_o + (warp * kRowsPerCta + g + 8) * kOPitch + c) = make_float2(o[n][2], o[n][3]);
        }
        if (t4 == 0) {
            sm_m[warp][g] = m_run[0];
            sm_m[warp][g + 8] = m_run[1];
            sm_l[warp][g] = l_run[0];
            sm_l[warp][g + 8] = l_run[1];
        }
    }
    __syncthreads();

    __shared__ float c_m[kMaxRowsPerCta];
    __shared__ float c_l[kMaxRowsPerCta];
    float* c_o = sm_o;   // [16][kOPitch]: combined in place over warp 0's slice (each element by its own thread)
    // merge weights, in the (now free) stage buffers after the warp partials: per row, each warp's
    // weight, each cluster peer's, the external partial's, and the output row offset
    float* s_f = sm_o + kWarps * kRowsPerCta * kOPitch;    // [kWarps][kMaxRowsPerCta]
    float* s_fp = s_f + kWarps * kMaxRowsPerCta;           // [kMaxClusterSplits][kMaxRowsPerCta]
    float* s_fe = s_fp + kMaxClusterSplits * kMaxRowsPerCta;
    int64_t* s_orow = reinterpret_cast<int64_t*>(s_fe + kMaxRowsPerCta);
    static_assert((kWarps * kRowsPerCta * kOPitch + (kWarps + kMaxClusterSplits + 1) * kMaxRowsPerCta) * 4 +
                          kMaxRowsPerCta * 8 <= kWarps * 2 * kSubBytes,
                  "merge scratch fits the stage buffers");
    // per row, once: the CTA's maximum and sum, and each warp's weight 2^(m_w - M)
    if (tid < nr) {
        const int r = tid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][r]);
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = fast_exp2(sm_m[w][r] - Ms);
            Ls = fmaf(sm_l[w][r], f, Ls);
            s_f[w * kMaxRowsPerCta + r] = f;
        }
        c_m[r] = M;
        c_l[r] = Ls;
    }
    __syncthreads();
    // the CTA's combined partial O, relative to its own row maxima
    auto combined4 = [&](int r, int c) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = s_f[w * kMaxRowsPerCta + r];
            const float4 v = *reinterpret_cast<const float4*>(sm_o + (w * kRowsPerCta + r) * kOPitch + c);
            o.x = fmaf(v.x, f, o.x);
            o.y = fmaf(v.y, f, o.y);
            o.z = fmaf(v.z, f, o.z);
            o.w = fmaf(v.w, f, o.w);
        }
        return o;
    };

    if constexpr (MERGE == kMergePush) {
        static_assert(NR != 32, "scoring-only tiles merge through the workspace");
        // CTAs 1 .. cs-1 send their combined partial into CTA 0's receive area with asynchronous remote
        // stores that count their bytes on CTA 0's barrier, and exit at once; CTA 0 announces the bytes
        // it expects, waits for them and merges alone.
        __shared__ __align__(16) float s_recv[kRecvFloats];   // [cs-1][nr][128] O, [cs-1][nr] m, [cs-1][nr] l
        const unsigned cs = cluster_size();
        const unsigned me = cluster_rank();
        const int npeer = (int)cs - 1;
        float* recv_m = s_recv + npeer * nr * kHeadDim;
        float* recv_l = recv_m + npeer * nr;
        cluster_wait_acquire();   // CTA 0's barrier is initialised
        if (me != 0) {
            const uint32_t rbar = cluster_map(&s_merge_bar, 0);
            const uint32_t dst = cluster_map(s_recv + (me - 1) * nr * kHeadDim, 0);
            for (int e = tid; e < nr * (kHeadDim / 4); e += kThreads)
                st_async_v4(dst + 16 * e, combined4(e >> 5, 4 * (e & 31)), rbar);
            if (tid < nr) {
                st_async_f32(cluster_map(recv_m + (me - 1) * nr + tid, 0), c_m[tid], rbar);
                st_async_f32(cluster_map(recv_l + (me - 1) * nr + tid, 0), c_l[tid], rbar);
            }
            return;
        }
        if (npeer > 0) {
            if (tid == 0) mbar_arrive_expect_tx(&s_merge_bar, (unsigned)(npeer * nr * (kHeadDim + 2) * 4));
            unsigned spins = 0;
            while (!mbar_try_wait_cluster(&s_merge_bar, 0)) {
                if (++spins == kSpinLimit) {
                    if (tid == 0) flag(p.err, FX_DEVERR_TIMEOUT);
                    break;
                }
            }
        }
        // per row, once: the weights of this CTA's warps, of each peer and of the external partial,
        // with the normalisation 1 / L folded in, and the output row's offset
        if (tid < nr) {
            const int r = tid;
            const float me_ = s_ext_m[r];
            float M = fmaxf(c_m[r], me_);
            for (int q = 0; q < npeer; ++q) M = fmaxf(M, recv_m[q * nr + r]);
            const float Ms = (M == -INFINITY) ? 0.f : M;
            const float a0 = fast_exp2(c_m[r] - Ms);
            const float ae = fast_exp2(me_ - Ms);
            float Ls = fmaf(c_l[r], a0, s_ext_l[r] * ae);
            for (int q = 0; q < npeer; ++q) {
                const float aq = fast_exp2(recv_m[q * nr + r] - Ms);
                Ls = fmaf(recv_l[q * nr + r], aq, Ls);
                s_fp[q * kMaxRowsPerCta + r] = aq;
            }
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s_f[w * kMaxRowsPerCta + r] *= a0 * inv;
            for (int q = 0; q < npeer; ++q) s_fp[q * kMaxRowsPerCta + r] *= inv;
            s_fe[r] = ae * inv;
            const int row = r0 + r;
            const int gi = row / p.Mq;
            const int i = row - gi * p.Mq;
            s_orow[r] = (((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7;
        }
        __syncthreads();
        const int c = tid;
#pragma unroll
        for (int r = 0; r < kExtRows; ++r) {
            if (r >= nr) break;
            float O = ext_oc[r] * s_fe[r];
#pragma unroll
            for (int w = 0; w < kWarps; ++w) O = fmaf(sm_o[(w * kRowsPerCta + r) * kOPitch + c], s_f[w * kMaxRowsPerCta + r], O);
            for (int q = 0; q < npeer; ++q) O = fmaf(s_recv[(q * nr + r) * kHeadDim + c], s_fp[q * kMaxRowsPerCta + r], O);
            p.out[s_orow[r] + c] = O;
        }
        return;
    }

    // pull and workspace merges start from the CTA's combined partial
    if (need_v) {
        for (int e = tid; e < nr * (kHeadDim / 4); e += kThreads) {
            const float4 o = combined4(e >> 5, 4 * (e & 31));
            *reinterpret_cast<float4*>(c_o + (e >> 5) * kOPitch + 4 * (e & 31)) = o;   // read above by this thread only
        }
    }

    if constexpr (MERGE == kMergePull) {
        // every split of this (b, h, row group) is one CTA of the cluster: merge through distributed
        // shared memory, each CTA producing a slice of the output rows
        static_assert(NR != 32, "scoring-only tiles merge through the workspace");
        cluster_sync();
        const unsigned cs = cluster_size();
        const unsigned me = cluster_rank();
        const int c = tid;
        int rn = (int)me;   // CTA q of the cluster produces rows q, q + cs, q + 2 cs, ...
#pragma unroll
        for (int r = 0; r < kExtRows; ++r) {
            if (r >= nr) break;
            if (r != rn) continue;
            rn += (int)cs;
            // one batch of independent remote loads, then the arithmetic
            float mq[kMaxClusterSplits], lq[kMaxClusterSplits], oq[kMaxClusterSplits];
#pragma unroll
            for (int q = 0; q < kMaxClusterSplits; ++q) {
                if ((unsigned)q < cs) {
                    mq[q] = ld_cluster(cluster_map(&c_m[r], q));
                    lq[q] = ld_cluster(cluster_map(&c_l[r], q));
                    oq[q] = ld_cluster(cluster_map(&c_o[r * kOPitch + c], q));
                } else {
                    mq[q] = -INFINITY;
                    lq[q] = 0.f;
                    oq[q] = 0.f;
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < kMaxClusterSplits; ++q) M = fmaxf(M, mq[q]);
            const float Ms = (M == -INFINITY) ? 0.f : M;
            float Ls = 0.f, O = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxClusterSplits; ++q) {
                const float w = fast_exp2(mq[q] - Ms);
                Ls = fmaf(lq[q], w, Ls);
                O = fmaf(oq[q], w, O);
            }
            const int row = r0 + r;
            const int gi = row / p.Mq;
            const int i = row - gi * p.Mq;
            p.out[((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + c] =
                finish_row(s_ext_m[r], s_ext_l[r], ext_oc[r], M, Ms, Ls, O);
        }
        cluster_sync();   // keep every CTA's shared memory alive until all reads are done
        return;
    }

    __syncthreads();
    for (int r = 0; r < nr; ++r) {
        const int64_t pi = (int64_t)(bh * p.R + r0 + r) * p.nsplit + split;
        if (need_v)
            for (int c = tid; c < kHeadDim; c += kThreads) p.part_o[pi * kHeadDim + c] = c_o[r * kOPitch + c];
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
#pragma unroll
    for (int r = 0; r < kExtRows; ++r) {
        if (r >= nr) break;
        const int row = r0 + r;
        const int64_t base = (int64_t)(bh * p.R + row) * p.nsplit;
        float M = -INFINITY;
        for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, __ldcg(p.part_m + base + s));
        const float Ms = (M == -INFINITY) ? 0.f : M;
        const int gi = row / p.Mq;
        const int i = row - gi * p.Mq;
        float* orow = p.out + ((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7);
        const int c = tid;
        float Ls = 0.f, O = 0.f;
        for (int s = 0; s < p.nsplit; ++s) {
            const float sc = fast_exp2(__ldcg(p.part_m + base + s) - Ms);
            Ls = fmaf(__ldcg(p.part_l + base + s), sc, Ls);
            O = fmaf(__ldcg(p.part_o + (base + s) * kHeadDim + c), sc, O);
        }
        orow[c] = finish_row(s_ext_m[r], s_ext_l[r], ext_oc[r], M, Ms, Ls, O);
    }
    if (tid == 0) p.counters[bh * p.nrg + rg] = 0u;
}

// Focal combine: merge split partials into the output rows and form the importance scores
//   s_j = sum_r exp2(t_rj - M_r) / Z_r   over the group's rows r, for cand_lo <= j < cand_hi.
__global__ void __launch_bounds__(256) focal_combine_kernel(const FocalCombineParams p)
{
    griddep_wait();   // the partials and logits come from the kernel just before
    griddep_launch();
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

template <int MODE, int MERGE, int NR>
cudaError_t launch_one(const AttnParams& p, bool pdl, cudaStream_t s)
{
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = attn_tile_kernel<MODE, MERGE, NR>;
    const bool cluster = MERGE != kMergeWorkspace;
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)attn_smem_bytes(NR, MODE));
        if (e != cudaSuccess) return e;
        if (cluster) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        configured = dev;
    }
    const size_t smem = attn_smem_bytes(NR, MODE);
    dim3 grid(p.nrg, p.nsplit, p.B * p.Hkv);
    // merged in a cluster: every split of one (b, h, row group) is one CTA of a (1, nsplit, 1) cluster
    return launch_kernel(kern, grid, dim3(kThreads), smem, s, pdl, cluster ? (unsigned)p.nsplit : 0u, p);
}

template <int MODE, int NR>
cudaError_t launch_rows(const AttnParams& p, bool pdl, cudaStream_t s)
{
    if constexpr (MODE == kModeFocal) {
        return launch_one<MODE, kMergeWorkspace, NR>(p, pdl, s);
    } else {
        const bool cl = p.nsplit <= kMaxClusterSplits;
        // pushed partials of the other CTAs must fit CTA 0's receive area
        const int rows = p.R < NR ? p.R : NR;
        const bool push = cl && (p.nsplit - 1) * rows * (kHeadDim + 2) <= kRecvFloats;
        if (push) return launch_one<MODE, kMergePush, NR>(p, pdl, s);
        return cl ? launch_one<MODE, kMergePull, NR>(p, pdl, s) : launch_one<MODE, kMergeWorkspace, NR>(p, pdl, s);
    }
}

template <int MODE>
cudaError_t launch_mode(const AttnParams& p, bool pdl, cudaStream_t s)
{
    if constexpr (MODE == kModeFocal) {
        if (p.rb == 32) return p.no_v ? launch_rows<MODE, 32>(p, pdl, s) : cudaErrorInvalidValue;
    }
    return p.rb == 8 ? launch_rows<MODE, 8>(p, pdl, s) : launch_rows<MODE, 16>(p, pdl, s);
}

}  // namespace

cudaError_t launch_attn_partial(const AttnParams& p, int mode, bool pdl, cudaStream_t s)
{
    if (p.rb != 8 && p.rb != 16 && p.rb != 32) return cudaErrorInvalidValue;
    if (mode == kModeFocal) return launch_mode<kModeFocal>(p, pdl, s);
    if (mode == kModeSparse) return launch_mode<kModeSparse>(p, pdl, s);
    return launch_mode<kModePrefix>(p, pdl, s);
}

cudaError_t launch_focal_combine(const FocalCombineParams& p, bool pdl, cudaStream_t s)
{
    const int ncand = p.scores ? (p.cand_hi - p.cand_lo) : 0;
    int gx = (ncand + 1023) / 1024;
    if (gx < 1) gx = 1;
    if (gx > 256) gx = 256;
    dim3 grid(gx, p.B * p.Hkv);
    return launch_kernel(focal_combine_kernel, grid, dim3(256), 0, s, pdl, 0u, p);
}

}  // namespace fx
