// Internal declarations shared by the libfx translation units (not part of the C ABI).
#pragma once

#include <cuda.h>   // CUtensorMap (the driver's encode function is resolved at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include <nvtx3/nvToolsExt.h>

#include "fx.h"

namespace fx {

constexpr int kHeadDim = 128;
constexpr int kMaxRows = 64;   // G * Mq limit per KV head
constexpr int kWarps = 4;                               // warps per attention CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kRowBytes = kHeadDim * 2;                 // one bf16 K or V row (256 bytes)
constexpr int kSub = 16;                                // keys per warp sub-tile (two n-tiles of S = Q K^T)
constexpr float kMaxSlack = 8.f;                       // online-softmax maximum slack (log2 units)
constexpr int kWarpStages = 3;                          // sub-tiles in flight per warp (at most)
constexpr int kRowsPerCta = 16;                         // query rows per CTA: one m16 MMA tile
constexpr int kPitch = kRowBytes + 16;                  // query tile row pitch: the 16-byte pad puts the 8
                                                        // rows of an ldmatrix on 8 distinct bank groups
constexpr int kKvPitch = kRowBytes;                     // staged K / V rows: unpadded, chunk-swizzled
constexpr int kSubBytes = 2 * kSub * kKvPitch;          // K and V rows of one sub-tile (8 KB)
constexpr int kTile = kWarps * kSub;                    // split lengths are multiples of this (whole sub-tiles per warp)
constexpr int kMaxSplitTokens = 4096;                   // gathered rows longer than 16 such splits merge in the workspace
constexpr unsigned kSpinLimit = 1u << 22;               // bounded mbarrier waits
constexpr int kMaxClusterSplits = 16;                   // splits merged inside one thread-block cluster
constexpr int kRecvFloats = 1024;                       // CTA 0's receive area for pushed partials (4 KB)
constexpr int kResidentPerSm = 2;                       // attention CTAs that fit one SM (shared memory)
// Streaming decode kernel (decode_stream.cu): kStreamProducers producer warps and kStreamConsumers
// consumer warps share a ring of at most kStreamMaxSlots sub-tile slots; its dynamic shared memory stays
// within kStreamSmemMax so that two CTAs (two consecutive calls) share an SM.
constexpr int kStreamConsumers = 4;
constexpr int kStreamProducers = 4;
constexpr int kStreamRows = 8;                          // query rows per KV head it serves (R <= 8)
constexpr int kStreamMaxSlots = 12;
constexpr size_t kStreamSmemMax = 110u * 1024u;
// Arrival counters of the last-CTA merge live in a fixed region at the start of every workspace
// (one slot per (b, h, row group); grid.z <= 65535 and at most 4 row groups), so no other data of
// any call ever overlaps them and they stay zero between calls.
constexpr size_t kCounterSlots = 65536u * 4u;
constexpr size_t kCounterBytes = kCounterSlots * sizeof(unsigned);

constexpr int kMaxRowsPerCta = 32;                      // query rows of the widest (scores-only) CTA
// Query-tile rows held in shared memory for a CTA of nr rows (16 at least: the 16-row MMA tile).
__host__ __device__ constexpr int attn_q_rows(int nr) { return nr > kRowsPerCta ? nr : kRowsPerCta; }
// Dynamic shared memory of one attention CTA: the query tile and each warp's ring of sub-tile buffers.


// Which key sequence an attention CTA walks.
enum AttnMode : int {
    kModeFocal = 0,   // all rows 0 .. len-1 of one cache, optional causal window
    kModeSparse = 1,  // idx[0..k) then tail_lo .. len-1
    kModePrefix = 2,  // prefix (dense or idx) ++ branch suffix ++ branch draft (causal)
};
// Sub-tiles in flight per warp: 3 for the decode and focal shapes (every CTA of a call resident at
// once, few sub-tiles per warp); 2 for shared-prefix verification, whose thousands of CTAs then fit
// three to an SM (measured: 8% faster verify, 20% slower decode with 2).
__host__ __device__ constexpr int attn_stages(int mode) { return mode == kModePrefix ? 2 : kWarpStages; }
inline size_t attn_smem_bytes(int nr, int mode)
{
    return 128 + (size_t)attn_q_rows(nr) * kPitch + (size_t)kWarps * attn_stages(mode) * kSubBytes;
}


struct AttnParams {
    // main cache (focal/sparse) or shared prefix (prefix mode: b-stride 0, len unused)
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* len;
    int64_t sb, sh, st;
    int B, Hkv, Tcap;
    // queries
    const uint16_t* q;
    int Hq, G, Mq, R;
    int q_pos0;     // focal: -1 or position of query 0
    float qscale;   // scale * log2(e): logits are kept in base-2 units
    // gathered rows: sparse idx [B, Hkv, kk] or prefix idx [Br, Hkv, kk]
    const int32_t* idx;
    int kk;
    int tail_lo;
    // prefix mode
    int P;
    const uint16_t* suf_k;
    const uint16_t* suf_v;
    int64_t suf_sh, suf_st;
    const int32_t* suf_off;
    const int32_t* suf_len;   // [Br] suffix rows (suf_off holds starts), or nullptr (suf_off[b+1] - suf_off[b])
    const int32_t* pre_len;   // [Br] visible prefix rows (fork positions), or nullptr (all P)
    // prefix mode: the dense prefix's partial (m, l, O) per row, computed by the tensor-core prefix
    // kernel ([Hkv][Br][R] rows) and folded into the final merge; nullptr when the prefix is in the keys
    const float* ext_m;
    const float* ext_l;
    const float* ext_o;
    int suf_rows, max_suffix;
    const uint16_t* dr_k;
    const uint16_t* dr_v;
    int64_t dr_sb, dr_si, dr_sh;
    // split geometry
    int nsplit, split_len, nrg, stages;
    int rb;         // query rows per CTA (8 or 16)
    int prefetch;   // lengths / indices / K-V rows may be read before the preceding kernel finishes
    int no_v;       // focal: scores only (no output rows), so V is neither read nor multiplied
    // outputs / scratch
    float* part_m;        // [B*Hkv*R*nsplit]
    float* part_l;        // [B*Hkv*R*nsplit]
    float* part_o;        // [B*Hkv*R*nsplit*128]
    float* logits;        // focal scores: [B*Hkv*R*Tcap] base-2 logits, or nullptr
    unsigned* counters;   // [B*Hkv*nrg] arrival counters for the last-CTA merge (sparse/prefix)
    float* out;           // [B, Hq, Mq, 128] fp32 (merged by the last CTA in sparse/prefix mode)
    unsigned* err;        // device error word
    unsigned spin_limit;  // polls of a bounded mbarrier wait before it gives up (kSpinLimit)
    unsigned test_stall;  // testing: polls of one extra wait on a barrier nothing arrives on (0: none)
    int tail_tma;         // streaming decode: contiguous tail rows come by TMA through the tensor maps
};

// Scores-only focal calls on the tensor cores (score_tc.cu): one persistent CTA per SM takes key ranges
// ("items") of score_item_tiles(N) tiles of kScoreKeys keys (N = score_tc_cols(rows), at most 64) and
// keeps kScoreBufs of them in flight, each range's logits in its own part of the tensor memory.
constexpr int kScoreKeys = 128;
constexpr int kScoreTmemCols = 512;   // the whole tensor memory of the SM
constexpr int kScoreBufs = 4;         // ranges in flight per CTA
constexpr int kScoreStages = 4;       // 32 KB K tiles in flight per CTA
__host__ __device__ constexpr int score_item_tiles(int n_cols) { return (kScoreTmemCols / kScoreBufs) / n_cols; }
// The N of a call with R rows: 16, 32 or 64 (each of the kernel's two row halves a power of two).
__host__ __device__ constexpr int score_tc_cols(int R) { return R <= 16 ? 16 : (R <= 32 ? 32 : 64); }

struct ScoreParams {
    const int32_t* len;       // [B], shared by the layers
    int B, Hkv, Tcap;
    int layers;               // layers scored in one launch; pairs = layers * B * Hkv
    int k_bcast;              // the cache has batch stride 0: the tensor map's batch extent is 1
    const uint16_t* q;        // [B, Hq, Mq, 128]
    int Hq, G, Mq, R;
    int q_pos0;
    float qscale;             // scale * log2(e)
    int pairs, nsplit, split_len;
    int cand_lo, cand_hi;
    float* part_m;            // [pairs][nsplit][R] row maximum of each key range
    float* part_l;            // [pairs][nsplit][R] row sum of each key range
    unsigned* counters;       // ticket, exit count, arrivals [pairs], then 8-byte words [pairs][R] of the merged
                              // c_r with a valid bit (all zero between calls)
    float* scores;            // [pairs][cand_hi - cand_lo]
    unsigned* err;
    unsigned spin_limit;
};

struct FocalCombineParams {
    const float* part_m;
    const float* part_l;
    const float* part_o;
    const float* logits;
    const int32_t* len;
    int B, Hkv, Tcap, Hq, G, Mq, R, nsplit;
    int cand_lo, cand_hi;
    float* out;
    float* scores;
    unsigned* err;
};

// Dense shared prefix on the tensor cores: the partial (m, l, O) of every (KV head, branch, row).
struct PrefixTcParams {
    const uint16_t* pk;
    const uint16_t* pv;
    int64_t p_sh, p_st;
    int P;
    const int32_t* pre_len;   // [Br] fork positions or nullptr
    const uint16_t* q;        // [Br, Hq, Mq, 128]
    int Br, Hkv, Hq, G, Mq, R;
    float qscale;
    float* ext_m;             // [Hkv][Br][R]
    float* ext_l;
    float* ext_o;             // [Hkv][Br][R][128]
    unsigned* err;
};

struct TopkParams {
    const float* scores;
    int rows, n, k;
    const int32_t* prev;
    int prev_early;   // prev may be read before the preceding kernel finishes (k <= 1024 only)
    int32_t* out;
    unsigned* err;
};

struct CompactParams {
    const uint16_t* sk;
    const uint16_t* sv;
    const int32_t* len;
    int64_t sb, sh, st, s_layer;
    int B, Hkv, Tcap;
    const int32_t* idx;
    int64_t idx_layer;   // element offset between the index sets of consecutive layers (0: shared)
    int kk, tail_lo;
    uint16_t* dk;
    uint16_t* dv;
    int32_t* dlen;
    int64_t db, dh, dt, d_layer;
    int dcap, n_layers, max_rows;
    unsigned* err;
};

struct AppendParams {
    uint16_t* k;
    uint16_t* v;
    int64_t sb, sh, st, layer;
    int B, Hkv, Tcap, n_layers;
    const uint16_t* k_new;   // [n_layers, B, Hkv, 128]
    const uint16_t* v_new;
    const int32_t* pos;      // [B]
    unsigned* err;
};

// An NVTX range over one library call, so that profiler timelines show each fx_* call by name (header-only
// NVTX v3: without a tool attached a push/pop costs a few nanoseconds).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Sets the calling thread's error message (read back by fx_last_error) and returns `st`.
fx_status set_error(fx_status st, const char* msg);

// Launchers.  `pdl`: launch as a programmatic dependent of the preceding kernel on the stream.
cudaError_t launch_attn_partial(const AttnParams& p, int mode, bool pdl, cudaStream_t s);
// Decode-shaped sparse calls (one query position, R <= 8): p.stages = ring slots, p.nsplit = splits.
// tk / tv: 4-D tensor maps of K and V ([B][Hkv][Tcap][128] bf16, boxes of 16 rows x 64 columns, 128-byte
// swizzle) when p.tail_tma, else unused.
cudaError_t launch_stream_decode(const AttnParams& p, const CUtensorMap* tk, const CUtensorMap* tv, bool pdl,
                                 cudaStream_t s);
// Encodes the tensor maps of a KV cache view for launch_stream_decode; false when the strides do not
// allow a tensor map (the kernel then copies the tail rows itself).
bool encode_kv_tensor_maps(const fx_kv_desc* kv, CUtensorMap* tk, CUtensorMap* tv);
size_t stream_decode_smem_bytes(int slots, int nsplit, int R);
cudaError_t launch_focal_combine(const FocalCombineParams& p, bool pdl, cudaStream_t s);
// tk: 5-D tensor map of K ([layers][B or 1][Hkv][Tcap][128] bf16, boxes of kScoreKeys rows x 64 columns);
// tq: 2-D tensor map of q ([layers B Hq Mq][128] bf16, boxes of N rows x 64 columns); both with the
// 128-byte swizzle.
cudaError_t launch_score_tc(const ScoreParams& p, const CUtensorMap* tk, const CUtensorMap* tq, int grid, bool pdl,
                            cudaStream_t s);
size_t score_tc_smem_bytes(int n_cols);
// Encodes the tensor maps for launch_score_tc (*bcast is set when the batch stride is 0); false when the
// strides or sizes allow no tensor map.
bool encode_score_maps(const fx_kv_desc* kv, int64_t layer_stride, int layers, const fx_bf16* q, int Hq, int Mq,
                       int n_cols, CUtensorMap* tk, CUtensorMap* tq, int* bcast);
cudaError_t launch_topk(const TopkParams& p, bool pdl, cudaStream_t s);
cudaError_t launch_prefix_tc(const PrefixTcParams& p, bool pdl, cudaStream_t s);
cudaError_t launch_focal_mass(const float* scores, int rows, int n, float inv_r, int accumulate, float* mass,
                              bool pdl, cudaStream_t s);
cudaError_t launch_compact(const CompactParams& p, bool pdl, cudaStream_t s);
cudaError_t launch_append(const AppendParams& p, bool pdl, cudaStream_t s);

// Launch `kern` with optional programmatic stream serialization and a (1, cluster_y, 1) cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          unsigned cluster_y, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_y > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = cluster_y;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

#ifdef __CUDACC__
// Programmatic dependent launch: wait until the preceding kernel on the stream has finished and its
// writes are visible (a no-op for a kernel launched without the attribute), and let the next kernel
// start launching.  Every kernel here triggers only after its own wait, so when a kernel starts,
// everything enqueued two or more launches before it has finished.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

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

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
#endif

// Query rows per attention CTA: 8 (keys on the MMA's M side) when at most 8 rows exist; for calls that
// only score (no output rows) and have more than 16 rows, 32 (keys on M, four query n-tiles); else 16.
inline int rows_per_block(int R, bool scores_only = false)
{
    if (R <= 8) return 8;
    if (scores_only && R > kRowsPerCta) return 32;
    return kRowsPerCta;
}

}  // namespace fx
