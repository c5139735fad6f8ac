// Scores-only focal calls on the tensor cores of sm_103a, with the logits kept in tensor memory.
//
// [FastKV] 2. Methodology, A. Token-Selective Propagation: a token's importance is the attention the
// window's query rows pay it, s_j = sum_r p_rj, where p_r is row r's softmax over every token it sees.
// [FastOCR] Methodology, Focal-Guided Pruning: the same sum over a focal layer's query rows.
//
// When many query rows share one key stream (G x Mq rows per KV head, e.g. 4 heads x 8 window
// positions) and no output rows are wanted, the split-KV path's fp32 logits are as large as K itself
// (R x 4 bytes per key against 256), and writing them out and reading them back doubles the call's
// traffic.  This kernel keeps them on chip.
//
// Work is cut into items: a contiguous range of 128 x (128 / N) keys of one (sequence, KV head), N = 16,
// 32 or 64 (the rows rounded up).  One persistent CTA per SM takes items from a ticket counter and keeps
// four in flight, each in its own quarter of the CTA's 512 tensor-memory columns (a "buffer"):
//   warp 0       draws the ticket and issues TMA copies of the item's K tiles (128 rows x 64 columns
//                each, 128-byte swizzle) into a ring of 32 KB slots shared by all items, the item's
//                query rows (an N-row K-major operand tile per buffer) with its first tile;
//   warp 1       (one thread) multiplies every tile as it lands,
//                  S^T = K Q^T   (M = 128 keys, N columns, K = 128 dims),
//                into the item's buffer, fp32, one N-column block per tile;
//   warps 2..9   (group A) read each tile's logits back as soon as its product is done (warp w reads
//                the keys of lane quarter w % 4, for half of the rows) and keep a running maximum and
//                sum per row and thread; after the last tile they reduce them to the item's (m, l) per
//                row and publish it;
//   warps 10..17 (group B, two subgroups of four taking alternate items) wait until every item of the
//                (sequence, KV head) has published; the first to claim the pair merges the rows' global
//                maximum M_r and sum Z_r once, in item order, and publishes c_r = M_r + log2 Z_r; then
//                each reads its item's logits once more and writes s_j = sum_r 2^(t_rj - c_r).
// A buffer is free for a new item once both groups and the product thread are done with it.  While
// the older items wait for their partners and form their scores, newer ones stream, so HBM stays busy.
// K is read once; the only other traffic is 2 R floats per item and the scores.
//
// Waiting for other items needs their CTAs to make progress.  Publishing an item (group A) waits only
// for its own products, never for another item, so an item that has been drawn always gets published.
// Tickets are drawn in order, and a CTA draws one only when a buffer is free, so it holds at most four
// items.  While the lowest incomplete (sequence, KV head) still has an undrawn item, every drawn item
// belongs to it or to an earlier one (those complete: all their items are drawn and get published); a
// CTA that cannot draw holds four of its items, so with nsplit <= 4 x (CTAs) some CTA can always draw
// the next one.  The host keeps nsplit at most twice the SM count.  Every wait is bounded all the same.
#include <cuda_bf16.h>
#include <stdint.h>

#include "attn_ptx.cuh"
#include "tc_ptx.cuh"

namespace fx {
namespace {

constexpr int kScAWarps = 8;   // group A: two warps per tensor-memory lane quarter (one per half of the rows)
constexpr int kScBWarps = 4;   // each of the two group-B subgroups: one warp per lane quarter
constexpr int kScCoordWarp = 2 + kScAWarps + 2 * kScBWarps;          // publishes each item's (m, l)
constexpr int kScThreads = 32 * (kScCoordWarp + 1);                  // + the copy warp and the product warp
constexpr int kScTileBytes = kScoreKeys * kRowBytes;   // one 128-key K tile (32 KB)
constexpr int kScHalf = kScTileBytes / 2;             // its 64-column half (one TMA copy)

__device__ __forceinline__ void tma_load_k(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                           uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Running (M, Z) of a softmax row: folds in a partial (m, l) = (maximum, sum of 2^(t - m)).
__device__ __forceinline__ void fold_partial(float& M, float& Z, float m, float l)
{
    if (m > M) {
        Z = Z * fast_exp2(M - m) + l;   // M = -inf at first: the product is 0
        M = m;
    } else if (m != -INFINITY) {
        Z = fmaf(l, fast_exp2(m - M), Z);
    }
}

// c_r = M_r + log2 Z_r (+inf when Z_r = 0) of rows r < R from nsplit partials pm/pl [nsplit][R], by kG
// threads (t = this thread's index), in a fixed order: thread t folds elements t, t + kG, ... (eight
// loads in flight at a time), then thread r < R folds the threads t = r (mod R) in order.  sync() is a
// barrier of the kG threads.
template <int kG, typename Sync>
__device__ __forceinline__ void merge_partials(const float* pm, const float* pl, int nsplit, int R, int t, float* s_m,
                                               float* s_z, float* c, Sync sync)
{
    const int nv = nsplit * R;
    if (kG % R == 0) {   // thread t meets row t % R only
        float M = -INFINITY, Z = 0.f;
        for (int u0 = t; u0 < nv; u0 += 16 * kG) {
            float mv[16], lv[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int u = u0 + k * kG;
                mv[k] = u < nv ? __ldcg(pm + u) : -INFINITY;
                lv[k] = u < nv ? __ldcg(pl + u) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 16; ++k) fold_partial(M, Z, mv[k], lv[k]);
        }
        s_m[t] = M;
        s_z[t] = Z;
        sync();
        if (t < R) {
            for (int u = t + R; u < kG; u += R) fold_partial(M, Z, s_m[u], s_z[u]);
            c[t] = Z > 0.f ? M + log2f(Z) : INFINITY;
        }
    } else if (t < R) {
        float M = -INFINITY, Z = 0.f;
        for (int s0 = 0; s0 < nsplit; s0 += 8) {
            float mv[8], lv[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int sp = s0 + k;
                mv[k] = sp < nsplit ? __ldcg(pm + sp * R + t) : -INFINITY;
                lv[k] = sp < nsplit ? __ldcg(pl + sp * R + t) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) fold_partial(M, Z, mv[k], lv[k]);
        }
        c[t] = Z > 0.f ? M + log2f(Z) : INFINITY;
    }
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float warp_max(float x)
{
    float y;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(y) : "f"(x));
    return y;
}

// Sums y[c] (c < H, H a power of two <= 32) over the 32 lanes of the warp: after log2(H) halving steps
// lane l holds the partial of row (l / (32 / H)) % H over the lanes that differ from it in the upper
// bits, and the remaining steps add across the lower bits, so every lane returns the total of that row.
template <int H>
__device__ __forceinline__ float warp_reduce_scatter(float (&y)[H], int lane)
{
    static_assert(H >= 1 && H <= 32 && (H & (H - 1)) == 0, "H must be a power of two <= 32");
    int nv = H;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (nv > 1) {
            const int half = nv / 2;
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int c = 0; c < H / 2; ++c) {
                if (c < half) {
                    const float keep = up ? y[c + half] : y[c];
                    const float send = up ? y[c] : y[c + half];
                    y[c] = keep + __shfl_xor_sync(kFull, send, o);
                }
            }
            nv = half;
        } else {
            y[0] += __shfl_xor_sync(kFull, y[0], o);
        }
    }
    return y[0];
}

// barrier of one epilogue group (named barrier 1: group A, 2: group B) of n threads
__device__ __forceinline__ void group_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// 8 K consecutive columns of this thread's tensor-memory lane (all loads in flight together), times `scale`
template <int K>
__device__ __forceinline__ void tmem_ld_cols(uint32_t addr, float scale, float (&v)[8 * K])
{
    uint32_t u[K][8];
#pragma unroll
    for (int c = 0; c < K; ++c) tmem_ld8_nowait(addr + (uint32_t)(8 * c), u[c]);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < K; ++c)
#pragma unroll
        for (int k = 0; k < 8; ++k) v[8 * c + k] = __uint_as_float(u[c][k]) * scale;
}

// S^T (tensor memory, 128 lanes x N columns) = K tile (smem) x Q tile (smem)^T over the 128 dims, as 8
// products of K = 16: a 16-element step is 32 bytes inside a 128-byte swizzled row, and steps 4..7 sit
// in the second 64-column block.
template <int N>
__device__ __forceinline__ void mma_kq(uint32_t d_tmem, uint32_t k_tile, uint32_t q_tile)
{
    constexpr uint32_t idesc = idesc_bf16(128, N, false);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint64_t da = sdesc(k_tile + (uint32_t)((ks >> 2) * kScHalf + (ks & 3) * 32));
        const uint64_t db = sdesc(q_tile + (uint32_t)((ks >> 2) * N * 128 + (ks & 3) * 32));
        const uint32_t acc = ks > 0 ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(da), "l"(db), "r"(idesc), "r"(acc));
    }
}

// One item: its (layer, sequence, KV head) -- the "pair" --, its key range [ja, jb) and the visible part
// [ja, jv).
struct Item {
    int pair, split, layer, b, h, ja, jb, jv, ntile;
    bool bad_len;
};

__device__ __forceinline__ Item decode_item(const ScoreParams& p, int item)
{
    Item it;
    it.pair = item / p.nsplit;
    it.split = item - it.pair * p.nsplit;
    const int per_layer = p.B * p.Hkv;
    it.layer = it.pair / per_layer;
    const int bh = it.pair - it.layer * per_layer;
    it.b = bh / p.Hkv;
    it.h = bh - it.b * p.Hkv;
    int lenb = p.len[it.b];
    it.bad_len = lenb < 0 || lenb > p.Tcap;
    if (it.bad_len) lenb = lenb < 0 ? 0 : p.Tcap;
    it.ja = it.split * p.split_len;
    it.jb = min(it.ja + p.split_len, p.Tcap);
    it.jv = max(it.ja, min(it.jb, lenb));
    it.ntile = (it.jv - it.ja + kScoreKeys - 1) / kScoreKeys;
    return it;
}

template <int NC2>   // N = 16 NC2 columns per tile
__global__ void __launch_bounds__(kScThreads, 1) score_tc_kernel(const ScoreParams p, const __grid_constant__ CUtensorMap tm_k,
                                                                   const __grid_constant__ CUtensorMap tm_q)
{
    constexpr int N = 16 * NC2;
    constexpr int H = 8 * NC2;                      // rows per group-A warp
    constexpr int kTiles = score_item_tiles(N);   // tiles per item
    constexpr int kItemCols = kTiles * N;            // tensor-memory columns per buffer
    constexpr int S = kScoreStages;
    constexpr int NB = kScoreBufs;                // items in flight: one tensor-memory buffer each
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char* ring = base;                                       // S K tiles
    unsigned char* sQ0 = base + (size_t)S * kScTileBytes;             // Q tiles of the NB buffers

    __shared__ __align__(8) uint64_t full_bar[S];           // a K tile has landed (TMA bytes)
    __shared__ __align__(8) uint64_t empty_bar[S];          // its product has read it (commit)
    __shared__ __align__(8) uint64_t item_bar[NB];          // a buffer's item and limits are staged
    __shared__ __align__(8) uint64_t tile_bar[NB][kTiles];  // a tile's product is in tensor memory (commit)
    __shared__ __align__(8) uint64_t free_bar[NB];          // a buffer's item is done (each group warp + the product thread)
    __shared__ __align__(8) uint64_t pub_bar[NB];           // group A has staged a buffer's (m, l) rows
    __shared__ __align__(8) uint64_t fin_bar;               // every product of this CTA is done (commit)
    __shared__ uint32_t s_tmem;
    __shared__ int s_item[NB];
    __shared__ float s_pm[NB][kMaxRows];    // an item's (m, l) per row, from group A to the coordinator warp
    __shared__ float s_pl[NB][kMaxRows];
    __shared__ int s_lim[NB][kMaxRows];     // keys j < s_lim[hf][r] are visible to row r in that buffer's item
    __shared__ float s_wm[kScAWarps][H];  // per group-A warp and row of its half: maximum, and sum relative to it
    __shared__ float s_wl[kScAWarps][H];
    __shared__ float s_c[2][kMaxRows];         // group B: c_r = M_r + log2 Z_r of the subgroup's current pair
    __shared__ float s_ra[2][32 * kScBWarps];  // group B: per-thread (M, Z) while merging
    __shared__ float s_ra2[2][32 * kScBWarps];
    __shared__ int s_last;
    __shared__ unsigned s_g;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    unsigned* const ticket_ctr = p.counters;
    unsigned* const exit_ctr = p.counters + 1;
    unsigned* const arrive = p.counters + 2;            // [pairs]
    // [pairs * R] words: a pair's c_r with bit 32 set once it is out (8-byte aligned after the arrivals)
    unsigned long long* const cword = reinterpret_cast<unsigned long long*>(p.counters + ((2 + p.pairs + 1) & ~1));
    const unsigned total = (unsigned)(p.pairs * p.nsplit);
    const unsigned spin = p.spin_limit;

    // Shared-memory barriers and the tensor memory first: they touch no global memory, so with a
    // programmatic dependent launch this overlaps the preceding kernel's tail.
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int x = 0; x < NB; ++x) {
            mbar_init(&item_bar[x], 1);
            mbar_init(&pub_bar[x], 1);
            mbar_init(&free_bar[x], kScAWarps + kScBWarps + 2);   // group A, the item's B subgroup, products, coordinator
            for (int t = 0; t < kTiles; ++t) mbar_init(&tile_bar[x][t], 1);
        }
        mbar_init(&fin_bar, 1);
        s_g = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                     "r"(kScoreTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;

    // Counters, lengths and queries may be written by the preceding kernel on the stream.
    griddep_wait();
    griddep_launch();

    if (warp == 0) {
        // ---- items and copies ---------------------------------------------------------------------
        unsigned g = 0;   // K tiles issued so far (ring position)
        for (int i = 0;; ++i) {
            const int hf = i % NB;
            if (i >= NB) mbar_wait_bounded(&free_bar[hf], (unsigned)((i / NB) - 1) & 1u, p.err, spin);
            unsigned tk = 0;
            if (lane == 0) tk = atomicAdd(ticket_ctr, 1u);
            tk = __shfl_sync(kFull, tk, 0);
            if (tk >= total) {
                // No items left (a ticket far past the end means the counters did not start at zero): an
                // end marker for this iteration, and for the next one, where the other group-B subgroup
                // looks.
                if (lane == 0) {
                    if (tk >= total + gridDim.x) flag(p.err, FX_DEVERR_TIMEOUT);
                    s_item[hf] = -1;
                    s_g = g;
                    mbar_arrive(&item_bar[hf]);
                }
                const int i2 = i + 1;
                const int hf2 = i2 % NB;
                if (i2 >= NB) mbar_wait_bounded(&free_bar[hf2], (unsigned)((i2 / NB) - 1) & 1u, p.err, spin);
                if (lane == 0) {
                    s_item[hf2] = -1;
                    mbar_arrive(&item_bar[hf2]);
                }
                break;
            }
            const Item it = decode_item(p, (int)tk);
            if (lane == 0 && it.bad_len && it.split == 0 && it.h == 0) flag(p.err, FX_DEVERR_LEN);
            // each row's visibility limit
            for (int r = lane; r < p.R; r += 32) {
                const int qi = r - (r / p.Mq) * p.Mq;
                int lim = it.jv;
                if (p.q_pos0 >= 0 && (int64_t)p.q_pos0 + qi + 1 < lim) lim = p.q_pos0 + qi + 1;
                s_lim[hf][r] = lim;
            }
            __syncwarp();
            if (lane == 0) {
                s_item[hf] = (int)tk;
                mbar_arrive(&item_bar[hf]);   // releases the limits and the item
                // The item's R query rows are rows ((layer B + b) Hq + h G) Mq .. + R - 1 of q viewed as
                // [layers B Hq Mq][128]:
                // they come with the first K tile, as the N-row K-major B operand of this buffer (the rows
                // past R belong to other items or lie past the end, and no result reads their columns).
                const int qrow = ((it.layer * p.B + it.b) * p.Hq + it.h * p.G) * p.Mq;
                const uint32_t dq = smem_addr(sQ0 + hf * N * kRowBytes);
                for (int t = 0; t < it.ntile; ++t, ++g) {
                    const unsigned s = g % S;
                    if (g >= (unsigned)S) mbar_wait_bounded(&empty_bar[s], ((g / S) - 1) & 1u, p.err, spin);
                    mbar_arrive_expect_tx(&full_bar[s], (unsigned)(kScTileBytes + (t == 0 ? N * kRowBytes : 0)));
                    if (t == 0) {
                        tma_load_2d(dq, &tm_q, 0, qrow, &full_bar[s]);
                        tma_load_2d(dq + N * 128, &tm_q, 64, qrow, &full_bar[s]);
                    }
                    const uint32_t dst = smem_addr(ring + (size_t)s * kScTileBytes);
                    const int j0 = it.ja + t * kScoreKeys;
                    const int cb = p.k_bcast ? 0 : it.b;
                    tma_load_k(dst, &tm_k, 0, j0, it.h, cb, it.layer, &full_bar[s]);
                    tma_load_k(dst + kScHalf, &tm_k, 64, j0, it.h, cb, it.layer, &full_bar[s]);
                }
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ---- products ------------------------------------------------------------------------------
        if (lane == 0) {
            unsigned g = 0;
            for (int i = 0;; ++i) {
                const int hf = i % NB;
                mbar_wait_bounded(&item_bar[hf], (unsigned)(i / NB) & 1u, p.err, spin);
                const int item = s_item[hf];
                if (item < 0) break;
                const Item it = decode_item(p, item);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dcol = tmem + (uint32_t)(hf * kItemCols);
                const uint32_t q = smem_addr(sQ0 + hf * N * kRowBytes);
                for (int t = 0; t < kTiles; ++t) {
                    if (t < it.ntile) {
                        const unsigned s = g % S;
                        mbar_wait_bounded(&full_bar[s], (g / S) & 1u, p.err, spin);
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        mma_kq<N>(dcol + (uint32_t)(t * N), smem_addr(ring + (size_t)s * kScTileBytes), q);
                        mma_commit(&empty_bar[s]);
                        ++g;
                    }
                    mma_commit(&tile_bar[hf][t]);   // every tile barrier completes once per use of the buffer
                }
                // this thread is past the item's barriers: the buffer's item and tile barriers may be re-armed
                // (its products are done once the epilogue has seen every tile barrier)
                mbar_arrive(&free_bar[hf]);
            }
            mma_commit(&fin_bar);
        }
    } else if (warp < 2 + kScAWarps) {
        // ---- group A: each tile's logits as soon as its product is done; the item's (m, l) per row ------
        const int a = warp - 2;                  // 0..7
        const int quarter = warp & 3;            // tensor-memory lanes: keys 32 quarter .. + 31 of a tile
        const int rh = a >> 2;                   // its rows: rh H .. rh H + H - 1
        const int kk = quarter * 32 + lane;      // this thread's key within a tile
        const int at = tid - 64;                 // 0 .. 255
        const float qs = p.qscale;
        for (int i = 0;; ++i) {
            const int hf = i % NB;
            const unsigned par = (unsigned)(i / NB) & 1u;
            mbar_wait_bounded(&item_bar[hf], par, p.err, spin);
            const int item = s_item[hf];
            if (item < 0) break;
            const Item it = decode_item(p, item);
            const uint32_t cbase =
                tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(hf * kItemCols + rh * H);
            int lim_min = it.jv;   // keys below it are visible to every row
            for (int r = 0; r < p.R; ++r) lim_min = min(lim_min, s_lim[hf][r]);
            // running maximum m and sum l = sum 2^(t - m) per row over this thread's keys; m moves only
            // when a logit exceeds it by more than kMaxSlack, so every term stays below 2^kMaxSlack
            float m[H], l[H];
#pragma unroll
            for (int c = 0; c < H; ++c) {
                m[c] = -INFINITY;
                l[c] = 0.f;
            }
            for (int t = 0; t < it.ntile; ++t) {
                mbar_wait_bounded(&tile_bar[hf][t], par, p.err, spin);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                __syncwarp();
                float v[H];   // raw products; the logit is v qs
                tmem_ld_cols<NC2>(cbase + (uint32_t)(t * N), 1.f, v);
                if (it.ja + (t + 1) * kScoreKeys <= lim_min) {
                    // every row sees this key (rows past R only feed unused columns): no per-row tests
                    float d[H];   // logit - m
                    bool grow = false;
#pragma unroll
                    for (int c = 0; c < H; ++c) {
                        d[c] = fmaf(v[c], qs, -m[c]);
                        grow |= d[c] > kMaxSlack;
                    }
                    if (grow) {   // the first tile, and rarely later: move the maxima that grew
#pragma unroll
                        for (int c = 0; c < H; ++c) {
                            if (d[c] > kMaxSlack) {
                                const float x = v[c] * qs;
                                l[c] *= fast_exp2(m[c] - x);
                                m[c] = x;
                                d[c] = 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int c = 0; c < H; ++c) l[c] += fast_exp2(d[c]);
                } else {
                    const int j = it.ja + t * kScoreKeys + kk;
#pragma unroll
                    for (int c = 0; c < H; ++c) {
                        const int r = rh * H + c;
                        if (r < p.R && j < s_lim[hf][r]) {
                            const float x = v[c] * qs;
                            if (x > m[c] + kMaxSlack) {
                                l[c] *= fast_exp2(m[c] - x);
                                m[c] = x;
                            }
                            l[c] += fast_exp2(x - m[c]);
                        }
                    }
                }
            }
            // this group is done with the buffer's tensor memory
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            // per warp: each row's maximum over the lanes, and the lanes' sums rescaled to it and added up
            // by a reduce-scatter (row rs_row(lane) ends in this lane); then over the four warps of each
            // row half: the item's (m, l) per row
            float y[H];
#pragma unroll
            for (int c = 0; c < H; ++c) {
                const float M = warp_max(m[c]);
                y[c] = m[c] == -INFINITY ? 0.f : l[c] * fast_exp2(m[c] - M);
                if (lane == 0) s_wm[a][c] = M;
            }
            const float ysum = warp_reduce_scatter<H>(y, lane);
            if ((lane & (32 / H - 1)) == 0) s_wl[a][(lane / (32 / H)) & (H - 1)] = ysum;
            group_sync(1, 32 * kScAWarps);
            if (at < p.R) {
                const int h2 = at / H;
                const int c = at - h2 * H;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < 4; ++w) M = fmaxf(M, s_wm[4 * h2 + w][c]);
                float L = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float mw = s_wm[4 * h2 + w][c];
                    if (mw != -INFINITY) L += s_wl[4 * h2 + w][c] * fast_exp2(mw - M);
                }
                s_pm[hf][at] = M;
                s_pl[hf][at] = L;
            }
            group_sync(1, 32 * kScAWarps);
            if (at == 0) mbar_arrive(&pub_bar[hf]);   // the coordinator warp publishes them
            if (lane == 0) mbar_arrive(&free_bar[hf]);
        }
    } else if (warp == kScCoordWarp) {
        // ---- coordinator: each item's (m, l) rows to global memory, then its arrival (release) ----------
        for (int i = 0;; ++i) {
            const int hf = i % NB;
            const unsigned par = (unsigned)(i / NB) & 1u;
            mbar_wait_bounded(&item_bar[hf], par, p.err, spin);
            const int item = s_item[hf];
            if (item < 0) break;
            const Item it = decode_item(p, item);
            mbar_wait_bounded(&pub_bar[hf], par, p.err, spin);
            const int64_t o = ((int64_t)it.pair * p.nsplit + it.split) * p.R;
            for (int r = lane; r < p.R; r += 32) {
                p.part_m[o + r] = s_pm[hf][r];
                p.part_l[o + r] = s_pl[hf][r];
            }
            __syncwarp();
            if (lane == 0) {
                red_release_add(&arrive[it.pair], 1u);   // releases the warp's stores of the partials
                mbar_arrive(&free_bar[hf]);
            }
        }
    } else {
        // ---- group B: the pair's merged (M_r, Z_r), then the item's scores; subgroup sg takes the items
        // i = sg (mod 2), so one subgroup's wait for a merge overlaps the other's work -------------------
        const int quarter = warp & 3;
        const int kk = quarter * 32 + lane;
        const int sg = (warp - 2 - kScAWarps) / kScBWarps;                // 0, 1
        const int bt = tid - 64 - 32 * (kScAWarps + sg * kScBWarps);      // 0 .. 127
        constexpr int kB = 32 * kScBWarps;
        const int bar = 2 + sg;
        float* const sc = s_c[sg];
        const float qs = p.qscale;
        const int ncand = p.cand_hi - p.cand_lo;
        for (int i = sg;; i += 2) {
            const int hf = i % NB;
            const unsigned par = (unsigned)(i / NB) & 1u;
            mbar_wait_bounded(&item_bar[hf], par, p.err, spin);
            const int item = s_item[hf];
            if (item < 0) break;
            const Item it = decode_item(p, item);
            const uint32_t cbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(hf * kItemCols);
            int lim_min = it.jv;
            for (int r = 0; r < p.R; ++r) lim_min = min(lim_min, s_lim[hf][r]);
            // the item's products are done (the last tile's commit follows all of them)
            if (it.ntile > 0) {
                mbar_wait_bounded(&tile_bar[hf][it.ntile - 1], par, p.err, spin);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                __syncwarp();
            }
            const int ca = max(it.ja, p.cand_lo);
            const int cb = min(it.jv, p.cand_hi);
            float* srow = p.scores + (int64_t)it.pair * ncand;
            if (it.split == 0) {
                // The pair's first item merges: once every item has published (arrive reaches nsplit), the
                // rows' c_r = M_r + log2 Z_r (+inf for a row that sees no key), folded in item order, go out
                // as one word per row with a valid bit, which the pair's other items poll.
                if (bt == 0) {
                    unsigned spins = 0;
                    while (ld_acquire_gpu(&arrive[it.pair]) < (unsigned)p.nsplit) {
                        if (++spins >= spin) {
                            flag(p.err, FX_DEVERR_TIMEOUT);
                            break;
                        }
                        __nanosleep(32);
                    }
                }
                group_sync(bar, kB);
                const int64_t prow = (int64_t)it.pair * p.nsplit * p.R;
                merge_partials<kB>(p.part_m + prow, p.part_l + prow, p.nsplit, p.R, bt, s_ra[sg], s_ra2[sg], sc,
                                   [bar] { group_sync(bar, kB); });
                group_sync(bar, kB);
                if (bt < p.R) st_relaxed_u64(cword + (int64_t)it.pair * p.R + bt, (1ull << 32) | __float_as_uint(sc[bt]));
            } else if (cb > ca && bt < p.R) {
                const unsigned long long* w = cword + (int64_t)it.pair * p.R + bt;
                unsigned long long x;
                unsigned spins = 0;
                while (((x = ld_relaxed_u64(w)) >> 32) == 0ull) {
                    if (++spins >= spin) {
                        flag(p.err, FX_DEVERR_TIMEOUT);
                        break;
                    }
                    __nanosleep(32);
                }
                sc[bt] = __uint_as_float((unsigned)x);
            }
            if (cb > ca) {
                group_sync(bar, kB);
                float ncr[N];   // -(M_r + log2 Z_r); -inf where the row sees nothing or r >= R
#pragma unroll
                for (int r = 0; r < N; ++r) ncr[r] = r < p.R ? -sc[r] : -INFINITY;
                // s_j = sum_r 2^(t_rj - M_r - log2 Z_r) for this thread's key of every tile
                for (int t = 0; t < it.ntile; ++t) {
                    const int j = it.ja + t * kScoreKeys + kk;
                    float v[N];
                    tmem_ld_cols<2 * NC2>(cbase + (uint32_t)(t * N), 1.f, v);
                    float acc0 = 0.f, acc1 = 0.f;
                    if (it.ja + (t + 1) * kScoreKeys <= lim_min) {
#pragma unroll
                        for (int r = 0; r < N; r += 2) {
                            acc0 += fast_exp2(fmaf(v[r], qs, ncr[r]));
                            acc1 += fast_exp2(fmaf(v[r + 1], qs, ncr[r + 1]));
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < N; r += 2) {
                            if (j < s_lim[hf][r]) acc0 += fast_exp2(fmaf(v[r], qs, ncr[r]));
                            if (j < s_lim[hf][r + 1]) acc1 += fast_exp2(fmaf(v[r + 1], qs, ncr[r + 1]));
                        }
                    }
                    if (ca <= j && j < cb) srow[j - p.cand_lo] = acc0 + acc1;
                }
            }
            // candidates of this item past the visible keys score 0
            {
                const int za = max(it.jv, p.cand_lo);
                const int zb = min(it.jb, p.cand_hi);
                for (int j = za + bt; j < zb; j += kB) srow[j - p.cand_lo] = 0.f;
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            group_sync(bar, kB);   // s_c may be rewritten for the next item
            if (lane == 0) mbar_arrive(&free_bar[hf]);
        }
    }

    // ---- the last CTA of the call resets the counters for the next call ----------------------------
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(exit_ctr, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (s_last) {
        for (int x = tid; x < p.pairs; x += kScThreads) arrive[x] = 0u;
        for (int x = tid; x < p.pairs * p.R; x += kScThreads) cword[x] = 0ull;
        if (tid == 0) {
            *ticket_ctr = 0u;
            *exit_ctr = 0u;
        }
    }
    // every copy has landed and every product is done before shared and tensor memory are released
    // (the waits return at once unless an earlier wait gave up)
    if (tid == 0) {
        const unsigned g = s_g;
        for (unsigned x = g > (unsigned)S ? g - S : 0u; x < g; ++x)
            mbar_wait_bounded(&full_bar[x % S], (x / S) & 1u, p.err, spin);
    }
    mbar_wait_bounded(&fin_bar, 0u, p.err, spin);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kScoreTmemCols));
}

template <int NC2>
cudaError_t launch_nc(const ScoreParams& p, const CUtensorMap* tk, const CUtensorMap* tq, int grid, bool pdl,
                      cudaStream_t s)
{
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = score_tc_smem_bytes(16 * NC2);
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<NC2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    const CUtensorMap mk = *tk;
    const CUtensorMap mq = *tq;
    return launch_kernel(score_tc_kernel<NC2>, dim3((unsigned)grid), dim3(kScThreads), smem, s, pdl, 0u, p, mk, mq);
}

}  // namespace

size_t score_tc_smem_bytes(int n_cols)
{
    // alignment pad, the ring and the query tiles of the buffers
    return 1024 + (size_t)kScoreStages * kScTileBytes + (size_t)kScoreBufs * n_cols * kRowBytes;
}

cudaError_t launch_score_tc(const ScoreParams& p, const CUtensorMap* tk, const CUtensorMap* tq, int grid, bool pdl,
                            cudaStream_t s)
{
    switch (score_tc_cols(p.R)) {
    case 16: return launch_nc<1>(p, tk, tq, grid, pdl, s);
    case 32: return launch_nc<2>(p, tk, tq, grid, pdl, s);
    case 64: return launch_nc<4>(p, tk, tq, grid, pdl, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fx
