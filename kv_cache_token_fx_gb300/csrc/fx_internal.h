// Internal declarations shared by the libfx translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fx.h"

namespace fx {

constexpr int kHeadDim = 128;
constexpr int kMaxRows = 64;   // G * Mq limit per KV head
constexpr int kWarps = 2;                               // warps per attention CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kRowBytes = kHeadDim * 2;                 // one bf16 K or V row (256 bytes)
constexpr int kTile = 32 * kWarps;                      // keys per tile: one key per thread
constexpr int kKPitch = kRowBytes + 16;                 // staged K row pitch: 16-byte pad keeps the
                                                        // lane-per-row 16-byte reads conflict-free
constexpr int kKStageBytes = kTile * kKPitch;           // 17 KB per staged tile of K
constexpr int kMaxSplitTokens = 4096;                   // longest split (bounds the index table)
constexpr unsigned kSpinLimit = 1u << 22;               // bounded mbarrier waits
constexpr int kMaxClusterSplits = 16;                   // splits merged inside one thread-block cluster
// Arrival counters of the last-CTA merge live in a fixed region at the start of every workspace
// (one slot per (b, h, row group); grid.z <= 65535 and at most 8 row groups), so no other data of
// any call ever overlaps them and they stay zero between calls.
constexpr size_t kCounterSlots = 65536u * 8u;
constexpr size_t kCounterBytes = kCounterSlots * sizeof(unsigned);

// Dynamic shared memory of one attention CTA: mbarriers, `stages` K tiles, the query rows (fp32)
// and the gathered-index table of its split.
inline size_t attn_smem_bytes(int stages, int rb, int gathered_split_len)
{
    return 128 + (size_t)stages * kKStageBytes + (size_t)rb * kHeadDim * sizeof(float) +
           (size_t)(gathered_split_len > 0 ? gathered_split_len : 0) * sizeof(int);
}

// Which key sequence an attention CTA walks.
enum AttnMode : int {
    kModeFocal = 0,   // all rows 0 .. len-1 of one cache, optional causal window
    kModeSparse = 1,  // idx[0..k) then tail_lo .. len-1
    kModePrefix = 2,  // prefix (dense or idx) ++ branch suffix ++ branch draft (causal)
};

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
    int suf_rows, max_suffix;
    const uint16_t* dr_k;
    const uint16_t* dr_v;
    int64_t dr_sb, dr_si, dr_sh;
    // split geometry
    int nsplit, split_len, nrg, stages;
    // outputs / scratch
    float* part_m;        // [B*Hkv*R*nsplit]
    float* part_l;        // [B*Hkv*R*nsplit]
    float* part_o;        // [B*Hkv*R*nsplit*128]
    float* logits;        // focal scores: [B*Hkv*R*Tcap] base-2 logits, or nullptr
    unsigned* counters;   // [B*Hkv*nrg] arrival counters for the last-CTA merge (sparse/prefix)
    float* out;           // [B, Hq, Mq, 128] fp32 (merged by the last CTA in sparse/prefix mode)
    unsigned* err;        // device error word
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

struct TopkParams {
    const float* scores;
    int rows, n, k;
    const int32_t* prev;
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
    int kk, tail_lo;
    uint16_t* dk;
    uint16_t* dv;
    int32_t* dlen;
    int64_t db, dh, dt, d_layer;
    int dcap, n_layers, max_rows;
    unsigned* err;
};

// Launchers (return cudaGetLastError() of the launch).
cudaError_t launch_attn_partial(const AttnParams& p, int mode, int rb, cudaStream_t s);
cudaError_t launch_focal_combine(const FocalCombineParams& p, cudaStream_t s);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t s);
cudaError_t launch_compact(const CompactParams& p, cudaStream_t s);

// Row-group width used for a given number of query rows per KV head.
inline int rows_per_block(int R) { return R <= 1 ? 1 : (R <= 2 ? 2 : (R <= 4 ? 4 : 8)); }

}  // namespace fx
