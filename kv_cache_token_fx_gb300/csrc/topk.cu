// Deterministic top-k per row for sm_103a: one CTA per row, radix select on the float bits.
//
// Order: score descending, index ascending (FastOCR, Focal-Guided Pruning: the top-attended tokens;
// ties go to the lower index).  Each fp32 score maps to a uint32 key that orders like the float.
// Four 8-bit radix passes find K*, the k-th largest key, and how many keys equal to K* must be taken
// (need_eq).  A final ordered pass -- a block-wide exclusive scan of (greater, equal) counts --
// writes every index with key > K* and the first need_eq indices with key == K*, in ascending index
// order.  No atomics decide the output, so the result is bit-reproducible.
//
// Warm start (FastOCR, Cross-Step Fixation Reuse): with the previous set S_prev, the threshold
// T = min over S_prev of the current scores is exceeded-or-met by at least k entries, so the top-k
// lies in {score >= T}; the radix passes only count those candidates.  The result is unchanged.
//
// Rows shorter than kClusterMinKeys are held in shared memory as keys.  Longer rows are split over a
// cluster of CTAs when there are few of them; otherwise each CTA reads its row from global memory until
// the remaining candidates fit in shared memory (rows up to kFilterMaxN), or on every pass (longer rows).
#include <stdint.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kSmemKeys = 44 * 1024;   // 176 KB of keys (plus 21 KB of static histogram rows)
constexpr int kClusterMinKeys = 16384;  // rows at least this long may be split over a cluster
constexpr int kClusterMaxCtasPerSm = 152;   // (times 2) cluster CTAs allowed in one launch

__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float f4_at(const float4& v, int c) { return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w; }

// Groups of 16 bytes when the row starts on a 16-byte boundary, else none (single scores only).
__device__ __forceinline__ int row_groups(const float* src, int n)
{
    return (reinterpret_cast<uintptr_t>(src) & 15u) == 0 ? n >> 2 : 0;
}

// skeys[j] = order_key(src[j]) for j < n, with 16-byte loads and stores when src is 16-byte aligned
// (skeys is).
__device__ __forceinline__ void load_keys(uint32_t* skeys, const float* src, int n)
{
    const int n4 = row_groups(src, n);
    const float4* s4 = reinterpret_cast<const float4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(skeys);
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kTkThreads) {
        const float4 v = __ldg(s4 + i);
        d4[i] = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
    }
    for (int j = 4 * n4 + threadIdx.x; j < n; j += kTkThreads) skeys[j] = order_key(__ldg(src + j));
}

template <bool SMEM>
__device__ __forceinline__ uint32_t get_key(const uint32_t* skeys, const float* src, int j)
{
    if (SMEM) return skeys[j];
    return order_key(__ldg(src + j));
}

// Block-wide exclusive scan of one uint32 per thread; returns the exclusive prefix, *total = sum.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* swarp, uint32_t* total)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) swarp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kTkWarps ? swarp[lane] : 0u;
        uint32_t winc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, winc, o);
            if (lane >= o) winc += t;
        }
        if (lane < kTkWarps) swarp[lane] = winc - w;   // exclusive warp offsets
        if (lane == kTkWarps - 1) swarp[32] = winc;    // block total
    }
    __syncthreads();
    const uint32_t res = swarp[warp] + inc - v;
    *total = swarp[32];
    __syncthreads();
    return res;
}

// Warp 0 (all 32 lanes): the radix digit that holds the krem-th largest counted key, from the 256-bin
// histogram, and the number of counted keys in higher bins; digit = 0xffffffff when fewer than krem
// keys were counted.
__device__ __forceinline__ void find_digit(const uint32_t* hist, uint32_t krem, uint32_t* digit, uint32_t* gt_out)
{
    const int lane = threadIdx.x & 31;
    uint32_t loc[8];
    uint32_t tot = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        loc[e] = hist[8 * lane + e];
        tot += loc[e];
    }
    uint32_t inc = tot;   // inclusive suffix sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, inc, o);
        if (lane + o < 32) inc += t;
    }
    const uint32_t all = __shfl_sync(0xffffffffu, inc, 0);
    uint32_t run = inc - tot;   // count of digits above this lane's bins
    int found = -1;
    uint32_t gt = 0u;
#pragma unroll
    for (int e = 7; e >= 0; --e) {
        const uint32_t before = run;
        run += loc[e];
        if (found < 0 && run >= krem && before < krem) {
            found = 8 * lane + e;
            gt = before;
        }
    }
    if (found >= 0) {
        *digit = (uint32_t)found;
        *gt_out = gt;
    }
    if (lane == 0 && all < krem) *digit = 0xffffffffu;   // fewer candidates than needed
}

struct SelectShared {
    uint32_t hist[256];
    uint32_t swarp[33];
    uint32_t digit, gt, thr, bad;
};

// Radix-digit counting.  Each lane counts with plain shared atomics into histogram row (lane mod 16),
// rows kHistStride = 257 words apart, and the rows are then added up per bin into hist[256].  Scores
// span few exponents, so most keys of a warp share one or two top-byte digits: with a row per lane
// pair, at most two lanes update one address, and lanes with the same digit hit different banks
// (257 = 1 mod 32).  Rows shared by whole warps let up to 32 lanes collide on one address.
constexpr int kHistRows = 16;
constexpr int kHistStride = 257;
constexpr int kHistWords = kHistRows * kHistStride;

__device__ __forceinline__ uint32_t* hist_row_of_lane(uint32_t* rows)
{
    return rows + (threadIdx.x & (kHistRows - 1)) * kHistStride;
}

__device__ __forceinline__ void hist_rows_clear(uint32_t* rows)
{
    for (int i = threadIdx.x; i < kHistWords; i += kTkThreads) rows[i] = 0u;
    __syncthreads();
}

// hist[b] = the sum of the rows' bin b; begins and ends with a barrier.
__device__ __forceinline__ void hist_rows_sum(const uint32_t* rows, uint32_t (*part)[256], uint32_t* hist)
{
    const int tid = threadIdx.x;
    __syncthreads();
    {
        const int b = tid & 255;
        const int g = tid >> 8;   // 4 groups of kHistRows / 4 rows
        uint32_t t = 0u;
#pragma unroll
        for (int r = 0; r < kHistRows / 4; ++r) t += rows[(g * (kHistRows / 4) + r) * kHistStride + b];
        part[g][b] = t;
    }
    __syncthreads();
    for (int b = tid; b < 256; b += kTkThreads) hist[b] = part[0][b] + part[1][b] + part[2][b] + part[3][b];
    __syncthreads();
}

// Counted: keys key_at(j), j = tid, tid + kTkThreads, ... < n, that are >= thr and equal prefix under
// pmask; the digit is byte `shift` of the key.  All threads call it; it begins and ends with a barrier.
template <typename KeyAt>
__device__ __forceinline__ void count_digits(KeyAt key_at, int n, uint32_t thr, uint32_t prefix, uint32_t pmask,
                                             int shift, uint32_t* rows, uint32_t (*part)[256], uint32_t* hist)
{
    const int tid = threadIdx.x;
    uint32_t* mine = hist_row_of_lane(rows);
    hist_rows_clear(rows);
    for (int j = tid; j < n; j += kTkThreads) {
        const uint32_t key = key_at(j);
        if (key >= thr && (key & pmask) == prefix) atomicAdd(&mine[(key >> shift) & 255u], 1u);
    }
    hist_rows_sum(rows, part, hist);
}

// The warm-start threshold: the smallest key over the previous set prow[0, k) (thread tid's first entry
// may have been read early into pre); 0 when an entry is out of [0, n) (reported once through err when
// report).  sh.thr must be 0xffffffff and sh.bad 0, visible to all threads, on entry; all threads call it.
constexpr int kNoPre = -2147483647 - 1;   // "prev index of this thread not loaded in advance"

template <typename KeyAt>
__device__ uint32_t warm_threshold(SelectShared& sh, const int32_t* prow, int pre, int k, int n, KeyAt key_at,
                                   unsigned* err, bool report)
{
    const int tid = threadIdx.x;
    uint32_t kmin = 0xffffffffu;
    for (int i = tid; i < k; i += kTkThreads) {
        const int t = (i == tid && pre != kNoPre) ? pre : prow[i];
        if (t < 0 || t >= n)
            sh.bad = 1u;
        else
            kmin = min(kmin, key_at(t));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    if ((tid & 31) == 0) atomicMin(&sh.thr, kmin);
    __syncthreads();
    if (sh.bad) {
        if (tid == 0 && report) atomicOr(err, FX_DEVERR_INDEX);
        return 0u;
    }
    return sh.thr;
}

// The top-k of one row of n keys (in skeys when SMEM, else read from src), written to orow in
// ascending index order.  prow: the previous set of this row (warm start) or nullptr.  All threads of
// the CTA call it; it begins and ends with a barrier.

template <bool SMEM>
__device__ void select_row(SelectShared& sh, uint32_t* hrows, uint32_t (*hpart)[256], const uint32_t* skeys,
                           const float* src, int n, int k, const int32_t* prow, int32_t* orow, unsigned* err,
                           int pre = kNoPre)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        sh.thr = prow != nullptr ? 0xffffffffu : 0u;
        sh.bad = 0u;
    }
    __syncthreads();

    // ---- warm-start threshold ----------------------------------------------------------------
    uint32_t thr = prow != nullptr ? warm_threshold(sh, prow, pre, k, n,
                                                    [&](int j) { return get_key<SMEM>(skeys, src, j); }, err, true)
                                   : 0u;

    // ---- radix select: K* and the number of equal keys to take --------------------------------
    uint32_t prefix = 0u, pmask = 0u;
    uint32_t krem = (uint32_t)k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int attempt = 0; attempt < 2; ++attempt) {
            count_digits([&](int j) { return get_key<SMEM>(skeys, src, j); }, n, thr, prefix, pmask, shift, hrows, hpart,
                         sh.hist);
            if (tid < 32) find_digit(sh.hist, krem, &sh.digit, &sh.gt);
            __syncthreads();
            if (sh.digit == 0xffffffffu && thr != 0u) {
                // only possible in pass 0 with a warm-start threshold built from repeated indices:
                // drop the threshold and count again
                thr = 0u;
                __syncthreads();
                continue;
            }
            break;
        }
        const bool missing = (sh.digit == 0xffffffffu);
        __syncthreads();
        if (missing) {
            // unreachable for 1 <= k <= n (checked on the host); keep the kernel finite anyway
            if (tid == 0) {
                atomicOr(err, FX_DEVERR_INDEX);
                sh.digit = 0u;
                sh.gt = 0u;
            }
            __syncthreads();
        }
        prefix |= sh.digit << shift;
        pmask |= 255u << shift;
        krem -= sh.gt;
        // When the chosen bin holds exactly the keys still needed, all of them are taken (not with a
        // warm-start threshold, which leaves keys of the bin below it uncounted).
        const bool all_taken = thr == 0u && sh.hist[sh.digit] == krem;
        __syncthreads();
        if (all_taken) break;
    }
    // the selected keys: masked key > prefix, and the first krem (in index order) with masked key == prefix
    const uint32_t kstar = prefix;
    const uint32_t need_eq = krem;

    // ---- ordered output -------------------------------------------------------------------------
    // position of an index j = (# greater before j) + min(# equal before j, need_eq); an equal key is
    // taken while (# equal before j) < need_eq (keys compared under pmask, the digits decided).
    // Positions are < k by construction; the bound checks keep a logic slip from writing past the row.
    if (SMEM) {
        // each thread owns a contiguous chunk of the row: one scan for the whole row
        const int per = (n + kTkThreads - 1) / kTkThreads;
        const int j0 = tid * per;
        const int j1 = min(n, j0 + per);
        uint32_t g = 0u, e = 0u;
        for (int j = j0; j < j1; ++j) {
            const uint32_t key = skeys[j] & pmask;
            g += key > kstar ? 1u : 0u;
            e += key == kstar ? 1u : 0u;
        }
        uint32_t total;
        const uint32_t ex = block_exclusive_scan(g | (e << 16), sh.swarp, &total);
        uint32_t gc = ex & 0xffffu;
        uint32_t ec = ex >> 16;
        for (int j = j0; j < j1; ++j) {
            const uint32_t key = skeys[j] & pmask;
            if (key > kstar) {
                const uint32_t pos = gc + min(ec, need_eq);
                if (pos < (uint32_t)k) orow[pos] = j;
                ++gc;
            } else if (key == kstar) {
                if (ec < need_eq && gc + ec < (uint32_t)k) orow[gc + ec] = j;
                ++ec;
            }
        }
    } else {
        // tiles of one key per thread (coalesced global reads), one scan per tile
        uint32_t base_g = 0u, base_e = 0u;
        for (int t0 = 0; t0 < n; t0 += kTkThreads) {
            const int j = t0 + tid;
            uint32_t g = 0u, e = 0u;
            if (j < n) {
                const uint32_t key = get_key<SMEM>(skeys, src, j) & pmask;
                g = key > kstar ? 1u : 0u;
                e = key == kstar ? 1u : 0u;
            }
            uint32_t total;
            const uint32_t ex = block_exclusive_scan(g | (e << 16), sh.swarp, &total);
            const uint32_t gc = base_g + (ex & 0xffffu);
            const uint32_t ec = base_e + (ex >> 16);
            if (g) {
                const uint32_t pos = gc + min(ec, need_eq);
                if (pos < (uint32_t)k) orow[pos] = j;
            } else if (e && ec < need_eq) {
                const uint32_t pos = gc + ec;
                if (pos < (uint32_t)k) orow[pos] = j;
            }
            base_g += total & 0xffffu;
            base_e += total >> 16;
        }
    }
    __syncthreads();
}

template <bool SMEM>
__global__ void __launch_bounds__(kTkThreads, 2) topk_kernel(const TopkParams p)
{
    extern __shared__ __align__(16) uint32_t skeys[];
    __shared__ SelectShared sh;
    __shared__ uint32_t s_rows[kHistWords];
    __shared__ uint32_t s_part[4][256];

    const int row = blockIdx.x;
    // this thread's entry of the previous set, read before the wait when the caller allows it
    int pre = kNoPre;
    if (p.prev_early && p.prev != nullptr && threadIdx.x < p.k) pre = p.prev[(int64_t)row * p.k + threadIdx.x];
    griddep_wait();   // the scores usually come from the kernel just before
    griddep_launch();
    const float* src = p.scores + (int64_t)row * p.n;
    if (SMEM) load_keys(skeys, src, p.n);
    select_row<SMEM>(sh, s_rows, s_part, skeys, src, p.n, p.k, p.prev != nullptr ? p.prev + (int64_t)row * p.k : nullptr,
                     p.out + (int64_t)row * p.k, p.err, pre);
}

// Few long rows: one cluster of kTkCluster CTAs per row.  CTA r of the cluster holds the contiguous
// chunk r of the row in shared memory; each radix pass counts the chunks in parallel, and every CTA
// adds the cluster's histograms through distributed shared memory and takes the same digit decision.  The ordered output offsets each chunk by the (greater, equal) counts of the chunks before
// it.  Same selection, bit for bit, as select_row.
constexpr int kTkCluster = 8;

__global__ void __launch_bounds__(kTkThreads, 2) topk_cluster_kernel(const TopkParams p)
{
    extern __shared__ __align__(16) uint32_t skeys[];   // this CTA's chunk
    __shared__ SelectShared sh;
    __shared__ uint32_t s_hist[2][256];   // this chunk's histogram, by round parity (read by the whole cluster)
    __shared__ uint32_t s_part[4][256];   // partial sums (of histogram rows, then of the cluster's chunks)
    __shared__ uint32_t s_rows[kHistWords];
    __shared__ uint32_t s_tot[256];       // the row's histogram
    __shared__ uint32_t s_cnt[2];         // (greater, equal) keys of this chunk
    __shared__ uint32_t s_base[2];
    const int row = blockIdx.y / kTkCluster;
    const unsigned me = cluster_rank();
    const int tid = threadIdx.x;
    const int n = p.n;
    const int k = p.k;
    const int chunk = (n + kTkCluster - 1) / kTkCluster;
    const int c0 = min(n, (int)me * chunk);
    const int cn = min(n, c0 + chunk) - c0;
    const int32_t* prow = p.prev != nullptr ? p.prev + (int64_t)row * k : nullptr;
    int pre = kNoPre;
    if (p.prev_early && prow != nullptr && tid < k) pre = prow[tid];
    griddep_wait();   // the scores usually come from the kernel just before
    griddep_launch();
    const float* src = p.scores + (int64_t)row * n;
    load_keys(skeys, src + c0, cn);
    if (tid == 0) {
        sh.thr = prow != nullptr ? 0xffffffffu : 0u;
        sh.bad = 0u;
    }
    __syncthreads();

    // warm-start threshold, the same in every CTA (scores read from global memory)
    uint32_t thr = prow != nullptr ? warm_threshold(sh, prow, pre, k, n, [&](int j) { return order_key(__ldg(src + j)); },
                                                    p.err, me == 0)
                                   : 0u;

    // Radix passes over 8-bit digits.  Each round every CTA counts its chunk into one of two histograms
    // (the other may still be read by a slower CTA), and after one cluster barrier every CTA adds up the
    // cluster's histograms in the same order and takes the same decision itself.
    uint32_t prefix = 0u, pmask = 0u;
    uint32_t krem = (uint32_t)k;
    int round = 0;
    bool all_taken = false;   // every counted key with the prefix is taken: no further pass is needed
    for (int pass = 0; pass < 4 && !all_taken; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t digit = 0u, gt = 0u;
        for (int attempt = 0; attempt < 2; ++attempt) {
            uint32_t* hist = s_hist[round & 1];
            ++round;
            count_digits([&](int j) { return skeys[j]; }, cn, thr, prefix, pmask, shift, s_rows, s_part, hist);
            cluster_sync();   // every chunk's histogram of this round is complete
            {
                // bin i, CTAs 2g and 2g + 1 of the cluster (integer sums: the order does not matter)
                const int i = tid & 255;
                const int g = tid >> 8;
                uint32_t t = 0u;
                for (int q = 2 * g; q < kTkCluster && q < 2 * g + 2; ++q) t += ld_cluster_u32(cluster_map(&hist[i], q));
                s_part[g][i] = t;
            }
            __syncthreads();
            for (int i = tid; i < 256; i += kTkThreads) s_tot[i] = s_part[0][i] + s_part[1][i] + s_part[2][i] + s_part[3][i];
            __syncthreads();
            if (tid < 32) find_digit(s_tot, krem, &sh.digit, &sh.gt);
            __syncthreads();
            digit = sh.digit;
            gt = sh.gt;
            if (digit == 0xffffffffu && thr != 0u) {
                thr = 0u;   // warm-start threshold from repeated indices: count again without it
                __syncthreads();
                continue;
            }
            break;
        }
        if (digit == 0xffffffffu) {
            // unreachable for 1 <= k <= n (checked on the host); keep the kernel finite anyway
            if (tid == 0 && me == 0) atomicOr(p.err, FX_DEVERR_INDEX);
            digit = 0u;
            gt = 0u;
        }
        prefix |= digit << shift;
        pmask |= 255u << shift;
        krem -= gt;
        // When the chosen bin holds exactly the keys still needed, all of them are taken (not with a
        // warm-start threshold, which leaves keys of the bin below it uncounted).
        all_taken = thr == 0u && s_tot[digit] == krem;
        __syncthreads();   // s_tot, sh.digit and sh.gt are rewritten in the next round
    }
    // the selected keys: masked key > prefix, and the first krem (in index order) with masked key == prefix
    const uint32_t kstar = prefix;
    const uint32_t need_eq = krem;

    // ordered output: counts of this chunk, then the offsets of the chunks before it
    const int per = (cn + kTkThreads - 1) / kTkThreads;
    const int j0 = tid * per;
    const int j1 = min(cn, j0 + per);
    uint32_t g = 0u, e = 0u;
    for (int j = j0; j < j1; ++j) {
        const uint32_t key = skeys[j] & pmask;
        g += key > kstar ? 1u : 0u;
        e += key == kstar ? 1u : 0u;
    }
    uint32_t total;
    const uint32_t ex = block_exclusive_scan(g | (e << 16), sh.swarp, &total);
    if (tid == 0) {
        s_cnt[0] = total & 0xffffu;
        s_cnt[1] = total >> 16;
    }
    cluster_sync();   // every chunk's counts are visible
    if (tid == 0) {
        uint32_t bg = 0u, be = 0u;
        for (unsigned q = 0; q < me; ++q) {
            bg += ld_cluster_u32(cluster_map(&s_cnt[0], q));
            be += ld_cluster_u32(cluster_map(&s_cnt[1], q));
        }
        s_base[0] = bg;
        s_base[1] = be;
    }
    __syncthreads();
    uint32_t gc = s_base[0] + (ex & 0xffffu);
    uint32_t ec = s_base[1] + (ex >> 16);
    int32_t* orow = p.out + (int64_t)row * k;
    for (int j = j0; j < j1; ++j) {
        const uint32_t key = skeys[j] & pmask;
        if (key > kstar) {
            const uint32_t pos = gc + min(ec, need_eq);
            if (pos < (uint32_t)k) orow[pos] = c0 + j;
            ++gc;
        } else if (key == kstar) {
            if (ec < need_eq && gc + ec < (uint32_t)k) orow[gc + ec] = c0 + j;
            ++ec;
        }
    }
    cluster_sync();   // keep every CTA's shared memory alive until all remote reads are done
}

// Many rows too long for shared memory: one CTA per row reads its scores from global memory (16-byte
// loads, four in flight per thread) on each radix pass, until the candidates -- the keys that match the
// digits chosen so far -- fit in shared memory.  The pass that finds them that few (the previous pass's
// chosen bin) also copies them there, (key, index), while it counts their next digit, and marks the keys
// above them -- all selected -- in a bitmap of the row; the remaining passes run on the copy.  The selected
// indices end as two bitmaps of the row (above K*, and equal to K* under the decided digits), and the
// ordered output is one block scan over them.  Same selection, bit for bit, as select_row.
constexpr int kFilterDynBytes = 200 * 1024;   // bitmaps + candidates (plus 21 KB of static histogram rows)
constexpr int kFilterMaxN = 1 << 18;          // two bitmaps of 32 KB at most

__host__ __device__ constexpr int filter_words(int n) { return (n + 31) / 32; }
__host__ __device__ constexpr int filter_cap(int n) { return (kFilterDynBytes - 8 * filter_words(n)) / 8; }

__device__ __forceinline__ void set_bit(uint32_t* bits, int j) { atomicOr(&bits[j >> 5], 1u << (j & 31)); }

// The 16-byte groups of a row held by one round: group i = r0 + u kTkThreads + tid (u < kRoundGroups)
// while i < n4; all loads of a round are in flight together.
constexpr int kRoundGroups = 4;

__device__ __forceinline__ void load_round(const float4* s4, int n4, int r0, float4 (&v)[kRoundGroups])
{
#pragma unroll
    for (int u = 0; u < kRoundGroups; ++u) {
        const int i = r0 + u * kTkThreads + threadIdx.x;
        v[u] = i < n4 ? __ldg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// f(key, j, valid) for every position of the row, in rounds that every thread of the CTA runs the same
// number of times (valid = false past the end), so that f may use warp-wide votes.
template <typename F>
__device__ __forceinline__ void for_each_key_global(const float* src, int n, F f)
{
    const int tid = threadIdx.x;
    const int n4 = row_groups(src, n);
    const float4* s4 = reinterpret_cast<const float4*>(src);
    for (int r0 = 0; r0 < n4; r0 += kRoundGroups * kTkThreads) {
        float4 v[kRoundGroups];
        load_round(s4, n4, r0, v);
#pragma unroll
        for (int u = 0; u < kRoundGroups; ++u) {
            const int i = r0 + u * kTkThreads + tid;
#pragma unroll
            for (int c = 0; c < 4; ++c) f(order_key(f4_at(v[u], c)), 4 * i + c, i < n4);
        }
    }
    for (int t0 = 4 * n4; t0 < n; t0 += kTkThreads) {
        const int j = t0 + tid;
        const bool ok = j < n;
        f(ok ? order_key(__ldg(src + j)) : 0u, j, ok);
    }
}

// The global pass that moves the candidates to shared memory.  Keys >= thr that match prefix under
// pmask: (key, index) appended to the candidates and, when COUNT, digit `shift` counted into this lane's
// histogram row `mine`; keys >= thr above the prefix (all selected): marked in gt_bits.  Without COUNT
// the prefix must be empty (every key >= thr is copied; mine and gt_bits are not used).  Candidate slots
// are reserved with one shared atomic per warp and round (4 kRoundGroups keys per lane), not one per key.
template <bool COUNT>
__device__ void collect_pass(const float* src, int n, uint32_t thr, uint32_t prefix, uint32_t pmask, int shift,
                             uint32_t* mine, uint32_t* gt_bits, uint32_t* ckey, int32_t* cidx, int cap,
                             uint32_t* ncand)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int n4 = row_groups(src, n);
    const float4* s4 = reinterpret_cast<const float4*>(src);
    auto visit = [&](uint32_t key, int j, bool ok) -> bool {
        const bool in = ok && key >= thr;
        if (!COUNT) return in;
        const uint32_t masked = key & pmask;
        const bool match = in && masked == prefix;
        if (match) atomicAdd(&mine[(key >> shift) & 255u], 1u);
        if (in && masked > prefix) set_bit(gt_bits, j);
        return match;
    };
    // cnt slots for this lane: a warp-inclusive scan and one atomic per warp; returns the lane's first slot
    auto reserve = [&](uint32_t cnt) -> uint32_t {
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t base = 0u;
        if (lane == 31 && wtot != 0u) base = atomicAdd(ncand, wtot);
        base = __shfl_sync(0xffffffffu, base, 31);
        return base + incl - cnt;
    };
    static_assert(4 * kRoundGroups <= 32, "one match bit per key of a round");
    auto put = [&](uint32_t slot, uint32_t key, int j) {
        if (slot < (uint32_t)cap) {
            ckey[slot] = key;
            cidx[slot] = j;
        }
    };
    for (int r0 = 0; r0 < n4; r0 += kRoundGroups * kTkThreads) {
        float4 v[kRoundGroups];
        load_round(s4, n4, r0, v);
        uint32_t m = 0u;
#pragma unroll
        for (int u = 0; u < kRoundGroups; ++u) {
            const int i = r0 + u * kTkThreads + tid;
#pragma unroll
            for (int c = 0; c < 4; ++c) m |= (uint32_t)visit(order_key(f4_at(v[u], c)), 4 * i + c, i < n4) << (4 * u + c);
        }
        uint32_t slot = reserve(__popc(m));
#pragma unroll
        for (int u = 0; u < kRoundGroups; ++u) {
            const int i = r0 + u * kTkThreads + tid;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if ((m >> (4 * u + c)) & 1u) put(slot++, order_key(f4_at(v[u], c)), 4 * i + c);
        }
    }
    for (int t0 = 4 * n4; t0 < n; t0 += kTkThreads) {
        const int j = t0 + tid;
        const bool ok = j < n;
        const uint32_t key = ok ? order_key(__ldg(src + j)) : 0u;
        const bool match = visit(key, j, ok);
        const uint32_t slot = reserve(match ? 1u : 0u);
        if (match) put(slot, key, j);
    }
}

// A threshold from a sample of the row: kSampleKeys keys at evenly spread positions (four consecutive
// keys per thread when the row is 16-byte aligned).  m = the expected number of the row's top k in the
// sample + 4 standard deviations + 8; the result is the lower edge of the 16-bit key bin that holds the
// sample's m-th largest key, so that with high probability at least k keys of the row reach it, and about
// m n / kSampleKeys do.  0 when that is not selective (m above half the sample) or the row is shorter than
// 4 kSampleKeys.  skey: scratch for kSampleKeys keys.  All threads call it; it ends with a barrier.
constexpr int kSampleKeys = 4 * kTkThreads;

__device__ __noinline__ uint32_t sample_threshold(const float* src, int n, int k, uint32_t* skey, SelectShared& sh, uint32_t* rows,
                                     uint32_t (*part)[256])
{
    const float mu = (float)kSampleKeys * (float)k / (float)n;
    const float mf = mu + 4.f * sqrtf(mu) + 8.f;
    if (n < 4 * kSampleKeys || mf > 0.5f * (float)kSampleKeys) return 0u;   // the same in every thread
    const int tid = threadIdx.x;
    const int n4 = row_groups(src, n);
    if (n4 > 0) {
        const int g = (int)(((int64_t)tid * n4) / kTkThreads);
        const float4 v = __ldg(reinterpret_cast<const float4*>(src) + g);
#pragma unroll
        for (int c = 0; c < 4; ++c) skey[4 * tid + c] = order_key(f4_at(v, c));
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) skey[4 * tid + c] = order_key(__ldg(src + ((int64_t)(4 * tid + c) * n) / kSampleKeys));
    }
    __syncthreads();
    uint32_t prefix = 0u, pmask = 0u;
    uint32_t krem = (uint32_t)ceilf(mf);
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = 24 - 8 * pass;
        count_digits([&](int j) { return skey[j]; }, kSampleKeys, 0u, prefix, pmask, shift, rows, part, sh.hist);
        if (tid < 32) find_digit(sh.hist, krem, &sh.digit, &sh.gt);
        __syncthreads();
        const uint32_t d = sh.digit;
        const uint32_t g = sh.gt;
        __syncthreads();   // sh.digit and sh.gt are rewritten by the next pass
        if (d == 0xffffffffu) return 0u;   // not reached: m <= half the sample
        prefix |= d << shift;
        pmask |= 255u << shift;
        krem -= g;
    }
    return prefix;
}

__global__ void __launch_bounds__(kTkThreads, 1) topk_filter_kernel(const TopkParams p)
{
    extern __shared__ __align__(16) uint32_t sdyn[];
    __shared__ SelectShared sh;
    __shared__ uint32_t s_rows[kHistWords];
    __shared__ uint32_t s_part[4][256];
    __shared__ uint32_t s_ncand;
    const int tid = threadIdx.x;
    const int row = blockIdx.x;
    const int n = p.n;
    const int k = p.k;
    const int nw = filter_words(n);
    const int cap = filter_cap(n);
    uint32_t* gt_bits = sdyn;
    uint32_t* eq_bits = sdyn + nw;
    uint32_t* ckey = sdyn + 2 * nw;
    int32_t* cidx = reinterpret_cast<int32_t*>(ckey + cap);
    uint32_t* mine = hist_row_of_lane(s_rows);
    const int32_t* prow = p.prev != nullptr ? p.prev + (int64_t)row * k : nullptr;
    int pre = kNoPre;
    if (p.prev_early && prow != nullptr && tid < k) pre = prow[tid];
    for (int i = tid; i < 2 * nw; i += kTkThreads) sdyn[i] = 0u;
    if (tid == 0) {
        sh.thr = prow != nullptr ? 0xffffffffu : 0u;
        sh.bad = 0u;
        s_ncand = 0u;
    }
    griddep_wait();   // the scores usually come from the kernel just before
    griddep_launch();
    const float* src = p.scores + (int64_t)row * n;
    __syncthreads();
    uint32_t thr = prow != nullptr ? warm_threshold(sh, prow, pre, k, n, [&](int j) { return order_key(__ldg(src + j)); },
                                                    p.err, true)
                                   : 0u;

    // A sampled threshold above the warm-start one lets the first pass copy its keys to shared memory
    // (when at least k and at most cap keys reach it; otherwise that pass is counted again without it).
    const uint32_t thr_s = sample_threshold(src, n, k, ckey, sh, s_rows, s_part);
    bool sampled = thr_s > thr;

    uint32_t prefix = 0u, pmask = 0u;
    uint32_t krem = (uint32_t)k;
    uint32_t bin = 0xffffffffu;   // counted keys that match the prefix (the last chosen bin)
    bool in_smem = false;
    int ncand = 0;
    bool all_taken = false;
    for (int pass = 0; pass < 4 && !all_taken; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int attempt = 0; attempt < 3; ++attempt) {
            bool overflow = false;
            if (in_smem) {
                count_digits([&](int j) { return ckey[j]; }, ncand, 0u, prefix, pmask, shift, s_rows, s_part, sh.hist);
            } else {
                if (pass == 0 && sampled) {
                    // copy the keys that reach the sampled threshold, then count their first digit there
                    collect_pass<false>(src, n, thr_s, 0u, 0u, shift, nullptr, nullptr, ckey, cidx, cap, &s_ncand);
                    __syncthreads();
                    const uint32_t got = s_ncand;
                    overflow = got > (uint32_t)cap;
                    ncand = (int)min(got, (uint32_t)cap);
                    in_smem = true;
                    count_digits([&](int j) { return ckey[j]; }, ncand, 0u, prefix, pmask, shift, s_rows, s_part,
                                 sh.hist);
                } else {
                    const bool collect = pass > 0 && bin <= (uint32_t)cap;
                    hist_rows_clear(s_rows);
                    if (collect) {
                        collect_pass<true>(src, n, thr, prefix, pmask, shift, mine, gt_bits, ckey, cidx, cap, &s_ncand);
                    } else {
                        for_each_key_global(src, n, [&](uint32_t key, int, bool ok) {
                            if (ok && key >= thr && (key & pmask) == prefix) atomicAdd(&mine[(key >> shift) & 255u], 1u);
                        });
                    }
                    hist_rows_sum(s_rows, s_part, sh.hist);
                    if (collect) {
                        const uint32_t got = s_ncand;
                        if (got != bin && tid == 0) atomicOr(p.err, FX_DEVERR_INDEX);   // a logic slip: keep the kernel finite
                        ncand = (int)min(got, (uint32_t)cap);
                        in_smem = true;
                    }
                }
            }
            if (tid < 32) find_digit(sh.hist, krem, &sh.digit, &sh.gt);
            __syncthreads();
            if (sampled && pass == 0 && (overflow || sh.digit == 0xffffffffu)) {
                // fewer than k keys, or more than the candidates' room, reached the sampled threshold: count
                // the row again without it (no bitmap bit was set: the prefix was empty)
                sampled = false;
                in_smem = false;
                ncand = 0;
                if (tid == 0) s_ncand = 0u;
                __syncthreads();
                continue;
            }
            if (sh.digit == 0xffffffffu && thr != 0u) {
                // only possible in pass 0 with a warm-start threshold built from repeated indices:
                // drop the threshold and count again
                thr = 0u;
                __syncthreads();
                continue;
            }
            break;
        }
        uint32_t digit = sh.digit;
        uint32_t gt = sh.gt;
        if (digit == 0xffffffffu) {
            // unreachable for 1 <= k <= n (checked on the host); keep the kernel finite anyway
            if (tid == 0) atomicOr(p.err, FX_DEVERR_INDEX);
            digit = 0u;
            gt = 0u;
        }
        prefix |= digit << shift;
        pmask |= 255u << shift;
        krem -= gt;
        bin = sh.hist[digit];
        // When the chosen bin holds exactly the keys still needed, all of them are taken: the counted ones,
        // which are exactly the copies in shared memory once the pass has copied them (keys below a
        // threshold are uncounted; they are below every copy), or every key of the bin without a threshold.
        all_taken = (thr == 0u || in_smem) && bin == krem;
        __syncthreads();   // sh.hist, sh.digit and sh.gt are rewritten in the next pass
    }
    // the selected keys: masked key > prefix, and the first krem (in index order) with masked key == prefix
    const uint32_t kstar = prefix;
    const uint32_t need_eq = krem;
    if (in_smem) {
        for (int c = tid; c < ncand; c += kTkThreads) {
            const uint32_t key = ckey[c] & pmask;
            if (key > kstar)
                set_bit(gt_bits, cidx[c]);
            else if (key == kstar)
                set_bit(eq_bits, cidx[c]);
        }
    } else {
        // no pass found few enough candidates (or the first pass decided): mark from the row itself.  A
        // key equal to K* under the decided digits is >= the warm-start threshold: K* is then a whole key.
        for_each_key_global(src, n, [&](uint32_t key, int j, bool ok) {
            const uint32_t masked = key & pmask;
            if (ok && masked > kstar)
                set_bit(gt_bits, j);
            else if (ok && masked == kstar)
                set_bit(eq_bits, j);
        });
    }
    __syncthreads();

    // ordered output: each thread owns a contiguous run of bitmap words; position of a selected index j =
    // (# greater before j) + min(# equal before j, need_eq), an equal one taken while (# equal before j) <
    // need_eq.  Positions are < k by construction; the bound checks keep a logic slip from writing past
    // the row.
    const int per = (nw + kTkThreads - 1) / kTkThreads;
    const int w0 = min(nw, tid * per);
    const int w1 = min(nw, w0 + per);
    uint32_t g = 0u, e = 0u;
    for (int w = w0; w < w1; ++w) {
        g += __popc(gt_bits[w]);
        e += __popc(eq_bits[w]);
    }
    uint32_t total;
    uint32_t gc = block_exclusive_scan(g, sh.swarp, &total);
    uint32_t ec = block_exclusive_scan(e, sh.swarp, &total);
    int32_t* orow = p.out + (int64_t)row * k;
    for (int w = w0; w < w1; ++w) {
        const uint32_t gw = gt_bits[w];
        const uint32_t ew = eq_bits[w];
        uint32_t u = gw | ew;
        while (u != 0u) {
            const int b = __ffs(u) - 1;
            u &= u - 1u;
            const int j = 32 * w + b;
            if ((gw >> b) & 1u) {
                const uint32_t pos = gc + min(ec, need_eq);
                if (pos < (uint32_t)k) orow[pos] = j;
                ++gc;
            } else {
                if (ec < need_eq && gc + ec < (uint32_t)k) orow[gc + ec] = j;
                ++ec;
            }
        }
    }
}

// Raise the kernel's dynamic shared memory limit to the largest key array (once per kernel and device).
template <auto KERN>
cudaError_t allow_smem_keys()
{
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device == dev) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemKeys * (int)sizeof(uint32_t));
    if (e == cudaSuccess) configured_device = dev;
    return e;
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, bool pdl, cudaStream_t s)
{
    // few long rows: a cluster of CTAs per row (about two CTAs per SM at most)
    if (p.n >= kClusterMinKeys && p.n <= kTkCluster * kSmemKeys && p.rows * kTkCluster <= 2 * kClusterMaxCtasPerSm) {
        const int chunk = (p.n + kTkCluster - 1) / kTkCluster;
        cudaError_t e = allow_smem_keys<topk_cluster_kernel>();
        if (e != cudaSuccess) return e;
        return launch_kernel(topk_cluster_kernel, dim3(1, p.rows * kTkCluster), dim3(kTkThreads),
                             (size_t)chunk * sizeof(uint32_t), s, pdl, (unsigned)kTkCluster, p);
    }
    // shorter rows: held in shared memory by one CTA per row.  Rows of kClusterMinKeys or more go to the
    // filtering kernel even when they would fit: measured on 1024 x 32760 (k = 2040), 141 us against
    // 329 us, since it works on about an eighth of the keys after two passes.
    if (p.n < kClusterMinKeys) {
        const size_t smem = (size_t)p.n * sizeof(uint32_t);
        cudaError_t e = allow_smem_keys<topk_kernel<true>>();
        if (e != cudaSuccess) return e;
        return launch_kernel(topk_kernel<true>, dim3(p.rows), dim3(kTkThreads), smem, s, pdl, 0u, p);
    }
    // many long rows: one CTA per row, finishing in shared memory once the candidates fit
    if (p.n <= kFilterMaxN) {
        static int configured_device = -1;
        int dev = 0;
        cudaGetDevice(&dev);
        if (configured_device != dev) {
            cudaError_t e = cudaFuncSetAttribute(topk_filter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kFilterDynBytes);
            if (e != cudaSuccess) return e;
            configured_device = dev;
        }
        const size_t smem = (size_t)8 * filter_words(p.n) + (size_t)8 * filter_cap(p.n);
        return launch_kernel(topk_filter_kernel, dim3(p.rows), dim3(kTkThreads), smem, s, pdl, 0u, p);
    }
    return launch_kernel(topk_kernel<false>, dim3(p.rows), dim3(kTkThreads), 0, s, pdl, 0u, p);
}

}  // namespace fx
