// Host side of libfx: argument checks, workspace planning, kernel launches and the device error word.
// Every entry point is extern "C" and declared in include/fx.h.
#include <math.h>

#include <algorithm>
#include <mutex>
#include <vector>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "fx_internal.h"

using namespace fx;

namespace {

constexpr int kAbiVersion = 3;
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

thread_local char g_msg[512] = "";

// Testing hook (fx_test_stall_wait): polls of one extra bounded wait that nothing completes.
unsigned g_test_stall = 0;

fx_status fail(fx_status st, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

fx_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(FX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

// Per-device error word written by the kernels (atomicOr of FX_DEVERR_* bits).
__device__ unsigned g_fx_device_error;

namespace {

struct DeviceState {
    bool ready = false;
    unsigned* err = nullptr;
    int sm_count = 0;
};
DeviceState g_dev[kMaxDevices];

fx_status device_state(DeviceState** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FX_ERR_CUDA, "device ordinal %d out of range", dev);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_fx_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        s.ready = true;
    }
    *out = &s;
    return FX_OK;
}

int sm_count_or_default()
{
    DeviceState* s = nullptr;
    if (device_state(&s) == FX_OK) return s->sm_count;
    return 152;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool row_stride_ok(int64_t s) { return s >= 0 && (s % 8) == 0; }
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int cdiv(int a, int b) { return (a + b - 1) / b; }

// Split-KV plan: how many query-row groups, how many key splits, how long each split is and how
// many staged K tiles each CTA keeps in flight.
struct Plan {
    int rb, nrg, nsplit, split_len, stages;
};

// `merge_in_cluster`: the splits of one (b, h, row group) are merged inside a thread-block cluster
// (sparse and prefix calls), which needs at most kMaxClusterSplits splits.  Gathered modes also keep
// each split within kMaxSplitTokens keys (the index table lives in shared memory).  Small calls get
// about two CTAs per SM in a single wave; large ones at least four full waves.
Plan make_plan(int pairs, int R, int max_keys, int sm_count, bool merge_in_cluster = false, bool gathered = false,
               bool scores_only = false)
{
    Plan pl;
    pl.rb = rows_per_block(R, scores_only);
    pl.nrg = cdiv(R, pl.rb);
    const int keys = max_keys > 0 ? max_keys : 1;
    const int per_split = pairs * pl.nrg;
    // Small calls: enough splits to give every SM work in one wave -- about one wave of resident CTAs
    // for the focal call; for calls merged in a cluster, about 1.5 CTAs per SM, because larger clusters
    // of large CTAs are harder to place (measured on the decode shapes: 4 splits of ~250 keys beat
    // 6, 8 and 16).  Large calls: at least four waves.
    const int resident = kResidentPerSm * sm_count;
    int ns;
    if (per_split >= resident)
        ns = cdiv(4 * resident, per_split);
    else if (merge_in_cluster)
        ns = std::min(resident / per_split, cdiv(3 * sm_count / 2, per_split));
    else
        ns = resident / per_split;
    const int min_ns = gathered ? cdiv(keys, kMaxSplitTokens) : 1;
    if (ns < min_ns) ns = min_ns;
    if (ns > cdiv(keys, 16)) ns = cdiv(keys, 16);
    if (merge_in_cluster && ns > kMaxClusterSplits && min_ns <= kMaxClusterSplits) ns = kMaxClusterSplits;
    if (ns < 1) ns = 1;
    pl.split_len = cdiv(cdiv(keys, ns), kTile) * kTile;   // equal whole sub-tiles per warp; the last split may be short
    pl.nsplit = cdiv(keys, pl.split_len);
    pl.stages = pl.split_len > kTile ? 2 : 1;
    return pl;
}

// Tensor-core scoring plan (scores-only calls with more than 8 rows): key ranges of as many whole
// 128-key tiles as one of a CTA's four tensor-memory buffers holds, spread evenly; one persistent CTA
// per SM (or per range, when there are fewer), and at most two ranges per SM per (b, h), so that the
// ranges of one (b, h) can always be in flight together.
struct ScoreTcPlan {
    int nsplit, split_len, grid;
};

bool make_score_tc_plan(int pairs, int R, int Tcap, int sm_count, ScoreTcPlan* sp)
{
    const int N = score_tc_cols(R);
    if (R > kMaxRows || Tcap < 1 || sm_count < 1) return false;
    const int cap = score_item_tiles(N) * kScoreKeys;
    const int ns = cdiv(Tcap, cap);
    if (ns > 2 * sm_count) return false;
    sp->split_len = cdiv(cdiv(Tcap, ns), kScoreKeys) * kScoreKeys;
    sp->nsplit = cdiv(Tcap, sp->split_len);
    const int64_t items = (int64_t)pairs * sp->nsplit;
    if (items > 0x7fffffff) return false;
    sp->grid = (int)std::min<int64_t>(items, sm_count);
    return true;
}

// Streaming decode plan: about 1.5 CTAs per SM per call (the splits of each (b, h) merged in a
// cluster) and as many ring slots as fit kStreamSmemMax, so that two CTAs share an SM and most of the
// next call's CTAs are resident, filling their rings, while this call finishes.  Measured on the
// FastOCR-shaped decode (64 (b, h) pairs, 718-973 keys): 3 splits beat 2 (fewer bytes in flight) and 4
// (the next call's CTAs find no room) at the early steps; rings of 8 slots with 3 CTAs per SM were
// slower than 12 slots with 2.
struct StreamPlan {
    int nsplit, slots;
};

StreamPlan make_stream_plan(int pairs, int R, int max_keys, int sm_count)
{
    int ns = pairs >= sm_count ? 1 : std::max(1, (3 * sm_count) / (2 * pairs));
    ns = std::min(ns, kMaxClusterSplits);
    ns = std::min(ns, std::max(1, cdiv(max_keys, kSub)));
    while (ns > 1 && stream_decode_smem_bytes(2 * kStreamProducers, ns, R) > kStreamSmemMax) --ns;
    int slots = (int)((kStreamSmemMax - stream_decode_smem_bytes(0, ns, R)) / kSubBytes);
    slots = std::min(slots, kStreamMaxSlots) / kStreamProducers * kStreamProducers;   // whole slots per producer
    return StreamPlan{ns, slots};
}

// cuTensorMapEncodeTiled, looked up once in the driver (the library does not link against it).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

struct Layout {
    size_t part_m, part_l, part_o, logits, counters, total;
};

Layout make_layout(int pairs, int R, const Plan& pl, int tcap_for_logits, bool with_counters)
{
    Layout L;
    const size_t P = (size_t)pairs * R * pl.nsplit;
    // every layout (even one that needs no counters) starts after the counter region, so a focal
    // call sharing the workspace can never overwrite the sparse/prefix arrival counters
    (void)with_counters;
    L.counters = 0;
    size_t off = kCounterBytes;
    L.part_m = off;
    off += round_up(P * sizeof(float));
    L.part_l = off;
    off += round_up(P * sizeof(float));
    L.part_o = off;
    off += round_up(P * kHeadDim * sizeof(float));
    L.logits = off;
    off += round_up((size_t)pairs * R * (size_t)(tcap_for_logits > 0 ? tcap_for_logits : 0) * sizeof(float));
    L.total = off;
    return L;
}

fx_status check_kv(const fx_kv_desc* kv, const char* name)
{
    if (!kv) return fail(FX_ERR_INVALID_ARG, "%s is NULL", name);
    if (!kv->k || !kv->v || !kv->len) return fail(FX_ERR_INVALID_ARG, "%s: k, v and len must be non-NULL", name);
    if (kv->d != kHeadDim) return fail(FX_ERR_UNSUPPORTED, "%s: head dim %d (only 128 is implemented)", name, kv->d);
    if (kv->B < 1 || kv->Hkv < 1 || kv->Tcap < 0)
        return fail(FX_ERR_INVALID_ARG, "%s: need B >= 1, Hkv >= 1, Tcap >= 0", name);
    if (!aligned16(kv->k) || !aligned16(kv->v))
        return fail(FX_ERR_INVALID_ARG, "%s: k and v must be 16-byte aligned", name);
    if (!row_stride_ok(kv->stride_b) || !row_stride_ok(kv->stride_h) || !row_stride_ok(kv->stride_t))
        return fail(FX_ERR_INVALID_ARG, "%s: strides must be non-negative multiples of 8 elements", name);
    return FX_OK;
}

fx_status check_heads(int Hq, int Hkv, int Mq)
{
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
        return fail(FX_ERR_INVALID_ARG, "Hq (%d) must be a positive multiple of Hkv (%d)", Hq, Hkv);
    if (Mq < 1) return fail(FX_ERR_INVALID_ARG, "Mq must be >= 1");
    if ((Hq / Hkv) * Mq > kMaxRows)
        return fail(FX_ERR_UNSUPPORTED, "G*Mq = %d query rows per KV head (at most %d)", (Hq / Hkv) * Mq, kMaxRows);
    return FX_OK;
}

fx_status check_ws(void* ws, size_t ws_bytes, size_t need)
{
    if (need == 0) return FX_OK;
    if (!ws) return fail(FX_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
        return fail(FX_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need) return fail(FX_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", ws_bytes, need);
    return FX_OK;
}

float log2e_scale(float scale) { return scale * 1.4426950408889634f; }

fx_status check_flags(unsigned flags)
{
    if (flags & ~(FX_LAUNCH_PDL | FX_LAUNCH_INPUTS_READY)) return fail(FX_ERR_INVALID_ARG, "unknown launch flags 0x%x", flags);
    return FX_OK;
}

}  // namespace

fx_status fx::set_error(fx_status st, const char* msg) { return fail(st, "%s", msg); }

extern "C" {

const char* fx_last_error(void) { return g_msg; }

int fx_abi_version(void) { return kAbiVersion; }

void fx_test_stall_wait(unsigned polls) { g_test_stall = polls; }

fx_status fx_device_errors(unsigned* bits, void* stream)
{
    if (!bits) return fail(FX_ERR_INVALID_ARG, "bits is NULL");
    DeviceState* ds = nullptr;
    fx_status st = device_state(&ds);
    if (st != FX_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned v = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(&v, ds->err, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
    e = cudaMemset(ds->err, 0, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
    *bits = v;
    return v ? FX_ERR_DEVICE : FX_OK;
}

fx_status fx_workspace_init(void* ws, size_t ws_bytes, void* stream)
{
    if (ws_bytes == 0) return FX_OK;
    if (!ws) return fail(FX_ERR_WORKSPACE, "workspace is NULL");
    cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
    return FX_OK;
}

// ---------------------------------------------------------------------------------------------
size_t fx_focal_workspace_bytes(int B, int Hkv, int Hq, int Mq, int Tcap)
{
    if (B < 1 || Hkv < 1 || Hq < Hkv || Mq < 1 || Tcap < 0) return 0;
    const int R = (Hq / Hkv) * Mq;
    // enough for both plans: with output rows, and scores only (which may use wider row groups)
    const Plan pl = make_plan(B * Hkv, R, Tcap, sm_count_or_default());
    const Plan ps = make_plan(B * Hkv, R, Tcap, sm_count_or_default(), false, false, true);
    return std::max(make_layout(B * Hkv, R, pl, Tcap, false).total, make_layout(B * Hkv, R, ps, Tcap, false).total);
}

// Workspace of the tensor-core scoring kernel over `layers` layers of B x Hkv pairs: the counter region,
// then the (m, l) partials of every key range; 0 when the kernel does not take the shape.
size_t score_tc_workspace_bytes(int layers, int B, int Hkv, int R, int Tcap, int sm_count)
{
    const int64_t pairs = (int64_t)layers * B * Hkv;
    ScoreTcPlan sp;
    if (R <= kStreamRows || pairs > 0x7fffffff || 4 + pairs + 2 * pairs * R > (int64_t)kCounterSlots ||
        !make_score_tc_plan((int)pairs, R, Tcap, sm_count, &sp))
        return 0;
    const size_t np = (size_t)pairs * sp.nsplit * R;
    return kCounterBytes + 2 * round_up(np * sizeof(float));
}

// Scores of `layers` consecutive layers (K of layer l at kv->k + l * layer_stride, its queries the l-th
// block of B Hq Mq rows of q, its scores the l-th block of B Hkv rows of cand_hi - cand_lo) on the
// tensor cores.  Returns false, launching nothing, when the kernel does not take the shape or K admits
// no tensor map; otherwise *st is the launch status.
bool score_tc_route(DeviceState* ds, const fx_kv_desc* kv, int64_t layer_stride, int layers, const fx_bf16* q,
                    int Hq, int Mq, int q_pos0, float scale, int cand_lo, int cand_hi, float* scores, void* ws,
                    size_t ws_bytes, bool pdl, cudaStream_t s, fx_status* st)
{
    const int G = Hq / kv->Hkv;
    const int R = G * Mq;
    const size_t need = score_tc_workspace_bytes(layers, kv->B, kv->Hkv, R, kv->Tcap, ds->sm_count);
    if (need == 0) return false;
    const int pairs = layers * kv->B * kv->Hkv;
    ScoreTcPlan sp;
    CUtensorMap tk, tq;
    int bcast = 0;
    if (!make_score_tc_plan(pairs, R, kv->Tcap, ds->sm_count, &sp) ||
        !encode_score_maps(kv, layer_stride, layers, q, Hq, Mq, score_tc_cols(R), &tk, &tq, &bcast))
        return false;
    if ((*st = check_ws(ws, ws_bytes, need)) != FX_OK) return true;
    const size_t np = (size_t)pairs * sp.nsplit * R;
    char* w = static_cast<char*>(ws);
    ScoreParams c;
    memset(&c, 0, sizeof c);
    c.len = kv->len;
    c.B = kv->B;
    c.Hkv = kv->Hkv;
    c.Tcap = kv->Tcap;
    c.layers = layers;
    c.k_bcast = bcast;
    c.q = q;
    c.Hq = Hq;
    c.G = G;
    c.Mq = Mq;
    c.R = R;
    c.q_pos0 = q_pos0;
    c.qscale = log2e_scale(scale);
    c.pairs = pairs;
    c.nsplit = sp.nsplit;
    c.split_len = sp.split_len;
    c.cand_lo = cand_lo;
    c.cand_hi = cand_hi;
    c.part_m = reinterpret_cast<float*>(w + kCounterBytes);
    c.part_l = reinterpret_cast<float*>(w + kCounterBytes + round_up(np * sizeof(float)));
    c.counters = reinterpret_cast<unsigned*>(w);
    c.scores = scores;
    c.err = ds->err;
    c.spin_limit = kSpinLimit;
    cudaError_t e = launch_score_tc(c, &tk, &tq, sp.grid, pdl, s);
    *st = e == cudaSuccess ? FX_OK : cuda_fail(e, "tensor-core scoring launch");
    return true;
}

fx_status fx_focal_attn_scores(const fx_kv_desc* kv, const fx_bf16* q, int Hq, int Mq, int q_pos0,
                               float scale, int cand_lo, int cand_hi, float* out, float* scores,
                               void* ws, size_t ws_bytes, unsigned flags, void* stream)
{
    fx::NvtxRange nvtx_range("fx_focal_attn_scores");
    fx_status st = check_kv(kv, "kv");
    if (st != FX_OK) return st;
    if ((st = check_flags(flags)) != FX_OK) return st;
    if ((st = check_heads(Hq, kv->Hkv, Mq)) != FX_OK) return st;
    if (!q || !aligned16(q)) return fail(FX_ERR_INVALID_ARG, "q must be non-NULL and 16-byte aligned");
    if (!out && !scores) return fail(FX_ERR_INVALID_ARG, "out and scores are both NULL");
    if (q_pos0 < -1) return fail(FX_ERR_INVALID_ARG, "q_pos0 must be -1 or >= 0");
    if (!isfinite(scale)) return fail(FX_ERR_INVALID_ARG, "scale must be finite");
    if (scores && (cand_lo < 0 || cand_lo > cand_hi || cand_hi > kv->Tcap))
        return fail(FX_ERR_INVALID_ARG, "candidate range [%d, %d) not inside [0, Tcap=%d]", cand_lo, cand_hi, kv->Tcap);
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FX_OK) return st;

    const int pairs = kv->B * kv->Hkv;
    const int G = Hq / kv->Hkv;
    const int R = G * Mq;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool pdl = (flags & FX_LAUNCH_PDL) != 0;

    // Scores only, more than 8 rows: the tensor-core kernel that keeps the logits on chip (its R fp32
    // logits per key would otherwise be written and read back), when K admits a tensor map.
    if (out == nullptr && score_tc_route(ds, kv, 0, 1, q, Hq, Mq, q_pos0, scale, cand_lo, cand_hi, scores, ws, ws_bytes,
                                         pdl, s, &st))
        return st;

    const Plan pl = make_plan(pairs, R, kv->Tcap, ds->sm_count, false, false, out == nullptr);
    const Layout L = make_layout(pairs, R, pl, kv->Tcap, false);
    if ((st = check_ws(ws, ws_bytes, L.total)) != FX_OK) return st;
    if (pairs > 65535 || pl.nsplit > 65535) return fail(FX_ERR_UNSUPPORTED, "grid too large");

    char* w = static_cast<char*>(ws);
    AttnParams p;
    memset(&p, 0, sizeof p);
    p.k = kv->k;
    p.v = kv->v;
    p.len = kv->len;
    p.sb = kv->stride_b;
    p.sh = kv->stride_h;
    p.st = kv->stride_t;
    p.B = kv->B;
    p.Hkv = kv->Hkv;
    p.Tcap = kv->Tcap;
    p.q = q;
    p.Hq = Hq;
    p.G = G;
    p.Mq = Mq;
    p.R = R;
    p.q_pos0 = q_pos0;
    p.qscale = log2e_scale(scale);
    p.nsplit = pl.nsplit;
    p.split_len = pl.split_len;
    p.nrg = pl.nrg;
    p.rb = pl.rb;
    p.stages = pl.stages;
    p.part_m = reinterpret_cast<float*>(w + L.part_m);
    p.part_l = reinterpret_cast<float*>(w + L.part_l);
    p.part_o = reinterpret_cast<float*>(w + L.part_o);
    p.logits = scores ? reinterpret_cast<float*>(w + L.logits) : nullptr;
    p.no_v = out == nullptr ? 1 : 0;
    p.err = ds->err;
    p.prefetch = (pdl && (flags & FX_LAUNCH_INPUTS_READY)) ? 1 : 0;
    cudaError_t e = launch_attn_partial(p, kModeFocal, pdl, s);
    if (e != cudaSuccess) return cuda_fail(e, "focal attention launch");

    FocalCombineParams c;
    c.part_m = p.part_m;
    c.part_l = p.part_l;
    c.part_o = p.part_o;
    c.logits = p.logits;
    c.len = kv->len;
    c.B = kv->B;
    c.Hkv = kv->Hkv;
    c.Tcap = kv->Tcap;
    c.Hq = Hq;
    c.G = G;
    c.Mq = Mq;
    c.R = R;
    c.nsplit = pl.nsplit;
    c.cand_lo = cand_lo;
    c.cand_hi = cand_hi;
    c.out = out;
    c.scores = scores;
    c.err = ds->err;
    e = launch_focal_combine(c, pdl, s);
    if (e != cudaSuccess) return cuda_fail(e, "focal combine launch");
    return FX_OK;
}

// ---------------------------------------------------------------------------------------------
fx_status fx_topk_select(const float* scores, int rows, int n, int k, const int32_t* prev_idx,
                         int32_t* idx_out, unsigned flags, void* stream)
{
    fx::NvtxRange nvtx_range("fx_topk_select");
    if (!scores || !idx_out) return fail(FX_ERR_INVALID_ARG, "scores and idx_out must be non-NULL");
    if (rows < 1) return fail(FX_ERR_INVALID_ARG, "rows must be >= 1");
    if (k < 1 || k > n) return fail(FX_ERR_INVALID_ARG, "need 1 <= k (%d) <= n (%d)", k, n);
    if (check_flags(flags) != FX_OK) return FX_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    fx_status st = device_state(&ds);
    if (st != FX_OK) return st;
    TopkParams p;
    p.scores = scores;
    p.rows = rows;
    p.n = n;
    p.k = k;
    p.prev = prev_idx;
    p.prev_early = (prev_idx && (flags & FX_LAUNCH_PDL) && (flags & FX_LAUNCH_INPUTS_READY)) ? 1 : 0;
    p.out = idx_out;
    p.err = ds->err;
    cudaError_t e = launch_topk(p, (flags & FX_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
    return FX_OK;
}

// ---------------------------------------------------------------------------------------------
fx_status fx_focal_mass(const float* scores, int rows, int n, int R, int accumulate, float* mass, unsigned flags,
                        void* stream)
{
    fx::NvtxRange nvtx_range("fx_focal_mass");
    if (!scores || !mass) return fail(FX_ERR_INVALID_ARG, "scores and mass must be non-NULL");
    if (rows < 1 || n < 1 || R < 1) return fail(FX_ERR_INVALID_ARG, "need rows, n, R >= 1");
    fx_status st = check_flags(flags);
    if (st != FX_OK) return st;
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FX_OK) return st;
    cudaError_t e = launch_focal_mass(scores, rows, n, 1.0f / (float)R, accumulate ? 1 : 0, mass,
                                      (flags & FX_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "focal mass launch");
    return FX_OK;
}

fx_status fx_csfr_schedule(int n_layers, const int32_t* focal_layers, int C, int first_step, int32_t* kind,
                           int32_t* src)
{
    if (!focal_layers || !kind || !src) return fail(FX_ERR_INVALID_ARG, "focal_layers, kind and src must be non-NULL");
    if (n_layers < 1 || C < 1 || C > n_layers) return fail(FX_ERR_INVALID_ARG, "need 1 <= C <= n_layers");
    for (int i = 0; i < C; ++i) {
        if (focal_layers[i] < 0 || focal_layers[i] >= n_layers)
            return fail(FX_ERR_INVALID_ARG, "focal layer %d out of range", focal_layers[i]);
        if (i > 0 && focal_layers[i] <= focal_layers[i - 1])
            return fail(FX_ERR_INVALID_ARG, "focal layers must be strictly ascending");
    }
    const int first = focal_layers[0];
    const int deepest = focal_layers[C - 1];
    int f = 0;   // focal layers at or before the current layer
    for (int l = 0; l < n_layers; ++l) {
        if (f < C && focal_layers[f] == l) {
            kind[l] = FX_CSFR_FOCAL;
            src[l] = l;
            ++f;
        } else if (l < first) {
            // before the first focal layer of this step: the deepest focal layer's set of the previous
            // step, or the whole cache when there is none yet
            kind[l] = first_step ? FX_CSFR_DENSE : FX_CSFR_PREVIOUS;
            src[l] = first_step ? -1 : deepest;
        } else {
            kind[l] = FX_CSFR_CURRENT;   // the nearest focal layer above, this step
            src[l] = focal_layers[f - 1];
        }
    }
    return FX_OK;
}

fx_status fx_choose_focal_layers(const float* ratio, int n_layers, int C, int32_t* layers_out)
{
    if (!ratio || !layers_out) return fail(FX_ERR_INVALID_ARG, "ratio and layers_out must be non-NULL");
    if (n_layers < 1 || C < 1 || C > n_layers) return fail(FX_ERR_INVALID_ARG, "need 1 <= C <= n_layers");
    for (int l = 0; l < n_layers; ++l)
        if (!isfinite(ratio[l])) return fail(FX_ERR_INVALID_ARG, "ratio[%d] is not finite", l);
    // the C largest ratios (ties: the lower layer), reported in ascending layer order
    std::vector<int> order(n_layers);
    for (int l = 0; l < n_layers; ++l) order[l] = l;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return ratio[a] > ratio[b]; });
    std::sort(order.begin(), order.begin() + C);
    for (int i = 0; i < C; ++i) layers_out[i] = order[i];
    return FX_OK;
}

// ---------------------------------------------------------------------------------------------
size_t fx_sparse_workspace_bytes(int B, int Hkv, int Hq, int k, int tail_lo, int Tcap)
{
    if (B < 1 || Hkv < 1 || Hq < Hkv || k < 0 || tail_lo < 0 || Tcap < 0) return 0;
    const int R = Hq / Hkv;
    if (R <= kStreamRows) return 0;   // the streaming kernel merges inside a cluster: no scratch
    const int max_keys = k + (Tcap > tail_lo ? Tcap - tail_lo : 0);
    const Plan pl = make_plan(B * Hkv, R, max_keys, sm_count_or_default(), true, k > 0);
    return make_layout(B * Hkv, R, pl, 0, true).total;
}

fx_status fx_sparse_gqa_decode(const fx_kv_desc* kv, const fx_bf16* q, int Hq, const int32_t* idx,
                               int k, int tail_lo, float scale, float* out, void* ws,
                               size_t ws_bytes, unsigned flags, void* stream)
{
    fx::NvtxRange nvtx_range("fx_sparse_gqa_decode");
    fx_status st = check_kv(kv, "kv");
    if (st != FX_OK) return st;
    if ((st = check_flags(flags)) != FX_OK) return st;
    if ((st = check_heads(Hq, kv->Hkv, 1)) != FX_OK) return st;
    if (!q || !aligned16(q)) return fail(FX_ERR_INVALID_ARG, "q must be non-NULL and 16-byte aligned");
    if (!out) return fail(FX_ERR_INVALID_ARG, "out is NULL");
    if (k < 0 || (k > 0 && !idx)) return fail(FX_ERR_INVALID_ARG, "need k >= 0 and idx when k > 0");
    if (tail_lo < 0) return fail(FX_ERR_INVALID_ARG, "tail_lo must be >= 0");
    if (!isfinite(scale)) return fail(FX_ERR_INVALID_ARG, "scale must be finite");
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FX_OK) return st;

    const int pairs = kv->B * kv->Hkv;
    const int G = Hq / kv->Hkv;
    const int R = G;
    const int max_keys = k + (kv->Tcap > tail_lo ? kv->Tcap - tail_lo : 0);
    const bool pdl = (flags & FX_LAUNCH_PDL) != 0;
    if (R <= kStreamRows) {
        // decode shapes: the streaming kernel (producer warp + CTA-wide ring, cluster merge)
        if (pairs > 65535) return fail(FX_ERR_UNSUPPORTED, "grid too large");
        const StreamPlan sp = make_stream_plan(pairs, R, max_keys, ds->sm_count);
        AttnParams p;
        memset(&p, 0, sizeof p);
        p.k = kv->k;
        p.v = kv->v;
        p.len = kv->len;
        p.sb = kv->stride_b;
        p.sh = kv->stride_h;
        p.st = kv->stride_t;
        p.B = kv->B;
        p.Hkv = kv->Hkv;
        p.Tcap = kv->Tcap;
        p.q = q;
        p.Hq = Hq;
        p.G = G;
        p.Mq = 1;
        p.R = R;
        p.q_pos0 = -1;
        p.qscale = log2e_scale(scale);
        p.idx = k > 0 ? idx : nullptr;
        p.kk = k;
        p.tail_lo = tail_lo;
        p.nsplit = sp.nsplit;
        p.stages = sp.slots;
        p.out = out;
        p.err = ds->err;
        p.spin_limit = kSpinLimit;
        p.test_stall = g_test_stall;
        p.prefetch = (pdl && (flags & FX_LAUNCH_INPUTS_READY)) ? 1 : 0;
        CUtensorMap tk, tv;
        p.tail_tma = encode_kv_tensor_maps(kv, &tk, &tv) ? 1 : 0;
        cudaError_t e = launch_stream_decode(p, &tk, &tv, pdl, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "sparse decode launch");
        return FX_OK;
    }
    const Plan pl = make_plan(pairs, R, max_keys, ds->sm_count, true, k > 0);
    const Layout L = make_layout(pairs, R, pl, 0, true);
    if ((st = check_ws(ws, ws_bytes, L.total)) != FX_OK) return st;
    if (pairs > 65535 || pl.nsplit > 65535) return fail(FX_ERR_UNSUPPORTED, "grid too large");

    char* w = static_cast<char*>(ws);
    AttnParams p;
    memset(&p, 0, sizeof p);
    p.k = kv->k;
    p.v = kv->v;
    p.len = kv->len;
    p.sb = kv->stride_b;
    p.sh = kv->stride_h;
    p.st = kv->stride_t;
    p.B = kv->B;
    p.Hkv = kv->Hkv;
    p.Tcap = kv->Tcap;
    p.q = q;
    p.Hq = Hq;
    p.G = G;
    p.Mq = 1;
    p.R = R;
    p.q_pos0 = -1;
    p.qscale = log2e_scale(scale);
    p.idx = k > 0 ? idx : nullptr;
    p.kk = k;
    p.tail_lo = tail_lo;
    p.nsplit = pl.nsplit;
    p.split_len = pl.split_len;
    p.nrg = pl.nrg;
    p.rb = pl.rb;
    p.stages = pl.stages;
    p.part_m = reinterpret_cast<float*>(w + L.part_m);
    p.part_l = reinterpret_cast<float*>(w + L.part_l);
    p.part_o = reinterpret_cast<float*>(w + L.part_o);
    p.counters = reinterpret_cast<unsigned*>(w + L.counters);
    p.out = out;
    p.err = ds->err;
    p.spin_limit = kSpinLimit;
    p.prefetch = (pdl && (flags & FX_LAUNCH_INPUTS_READY)) ? 1 : 0;
    cudaError_t e = launch_attn_partial(p, kModeSparse, pdl, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse decode launch");
    return FX_OK;
}

// ---------------------------------------------------------------------------------------------
fx_status fx_kv_compact(const fx_kv_desc* src, int64_t src_stride_layer, const int32_t* idx,
                        int64_t idx_stride_layer, int k, int tail_lo, const fx_kv_out_desc* dst,
                        int64_t dst_stride_layer, int n_layers, unsigned flags, void* stream)
{
    fx::NvtxRange nvtx_range("fx_kv_compact");
    fx_status st = check_kv(src, "src");
    if (st != FX_OK) return st;
    if ((st = check_flags(flags)) != FX_OK) return st;
    if (!dst) return fail(FX_ERR_INVALID_ARG, "dst is NULL");
    fx_kv_desc dview = {dst->k, dst->v, dst->len, dst->stride_b, dst->stride_h, dst->stride_t,
                        dst->B, dst->Hkv, dst->Tcap, dst->d};
    if ((st = check_kv(&dview, "dst")) != FX_OK) return st;
    if (dst->B != src->B || dst->Hkv != src->Hkv)
        return fail(FX_ERR_INVALID_ARG, "src and dst must have the same B and Hkv");
    if (n_layers < 1) return fail(FX_ERR_INVALID_ARG, "n_layers must be >= 1");
    if (k < 0 || (k > 0 && !idx)) return fail(FX_ERR_INVALID_ARG, "need k >= 0 and idx when k > 0");
    if (tail_lo < 0) return fail(FX_ERR_INVALID_ARG, "tail_lo must be >= 0");
    if (idx_stride_layer < 0) return fail(FX_ERR_INVALID_ARG, "idx_stride_layer must be >= 0");
    if (!row_stride_ok(src_stride_layer) || !row_stride_ok(dst_stride_layer))
        return fail(FX_ERR_INVALID_ARG, "layer strides must be non-negative multiples of 8 elements");
    if ((int64_t)src->B * n_layers > 65535 || src->Hkv > 65535) return fail(FX_ERR_UNSUPPORTED, "grid too large");
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FX_OK) return st;

    CompactParams p;
    p.sk = src->k;
    p.sv = src->v;
    p.len = src->len;
    p.sb = src->stride_b;
    p.sh = src->stride_h;
    p.st = src->stride_t;
    p.s_layer = src_stride_layer;
    p.B = src->B;
    p.Hkv = src->Hkv;
    p.Tcap = src->Tcap;
    p.idx = k > 0 ? idx : nullptr;
    p.idx_layer = idx_stride_layer;
    p.kk = k;
    p.tail_lo = tail_lo;
    p.dk = dst->k;
    p.dv = dst->v;
    p.dlen = dst->len;
    p.db = dst->stride_b;
    p.dh = dst->stride_h;
    p.dt = dst->stride_t;
    p.d_layer = dst_stride_layer;
    p.dcap = dst->Tcap;
    p.n_layers = n_layers;
    const int max_rows = k + (src->Tcap > tail_lo ? src->Tcap - tail_lo : 0);
    p.max_rows = max_rows < dst->Tcap ? max_rows : dst->Tcap;
    p.err = ds->err;
    cudaError_t e = launch_compact(p, (flags & FX_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "compaction launch");
    return FX_OK;
}

fx_status fx_kv_append(const fx_kv_out_desc* cache, int64_t stride_layer, int n_layers, const fx_bf16* k_new,
                       const fx_bf16* v_new, const int32_t* pos, unsigned flags, void* stream)
{
    fx::NvtxRange nvtx_range("fx_kv_append");
    fx_status st;
    if (!cache) return fail(FX_ERR_INVALID_ARG, "cache is NULL");
    if (!pos) return fail(FX_ERR_INVALID_ARG, "pos is NULL");
    fx_kv_desc view = {cache->k, cache->v, pos, cache->stride_b, cache->stride_h, cache->stride_t,
                       cache->B, cache->Hkv, cache->Tcap, cache->d};
    if ((st = check_kv(&view, "cache")) != FX_OK) return st;
    if ((st = check_flags(flags)) != FX_OK) return st;
    if (n_layers < 1) return fail(FX_ERR_INVALID_ARG, "n_layers must be >= 1");
    if (!k_new || !v_new) return fail(FX_ERR_INVALID_ARG, "k_new and v_new are required");
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
        return fail(FX_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (!row_stride_ok(stride_layer)) return fail(FX_ERR_INVALID_ARG, "stride_layer must be a non-negative multiple of 8 elements");
    // the append kernel copies 8 rows per CTA and its grid.x stays below 2^31
    if ((int64_t)n_layers * cache->B * cache->Hkv > (int64_t)0x7fffffff * 8)
        return fail(FX_ERR_UNSUPPORTED, "too many rows");
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FX_OK) return st;
    AppendParams p;
    p.k = cache->k;
    p.v = cache->v;
    p.sb = cache->stride_b;
    p.sh = cache->stride_h;
    p.st = cache->stride_t;
    p.layer = stride_layer;
    p.B = cache->B;
    p.Hkv = cache->Hkv;
    p.Tcap = cache->Tcap;
    p.n_layers = n_layers;
    p.k_new = k_new;
    p.v_new = v_new;
    p.pos = pos;
    p.err = ds->err;
    cudaError_t e = launch_append(p, (flags & FX_LAUNCH_PDL) != 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return FX_OK;
}

// ---------------------------------------------------------------------------------------------
// Layers are scored kRetainBatch at a time into their own score rows -- by one launch of the tensor-core
// scoring kernel over all of them when it takes the shape, so that one layer's last key ranges overlap
// the next layer's stream --, then selected by one top-k launch over all of them (many rows in flight
// hide each row's latency).  Measured on 32 layers of 4 x 8 x 32768 keys: batches of 8, 16 and 32
// layers took 2.34, 2.31 and 2.24 ms.
constexpr int kRetainBatch = 32;

size_t retain_scoring_bytes(int B, int Hkv, int Hq, int Mq, int Tcap)
{
    const size_t f = fx_focal_workspace_bytes(B, Hkv, Hq, Mq, Tcap);
    if (f == 0) return 0;
    const int R = (Hq / Hkv) * Mq;
    return round_up(std::max(f, score_tc_workspace_bytes(kRetainBatch, B, Hkv, R, Tcap, sm_count_or_default())));
}

size_t fx_retain_workspace_bytes(int B, int Hkv, int Hq, int Mq, int Tcap, int cand_hi)
{
    const size_t f = retain_scoring_bytes(B, Hkv, Hq, Mq, Tcap);
    if (f == 0 || cand_hi < 1) return 0;
    return f + round_up((size_t)kRetainBatch * B * Hkv * cand_hi * sizeof(float));
}

fx_status fx_kv_retain_per_layer(const fx_kv_desc* kv, int64_t src_stride_layer, int n_layers, const fx_bf16* q,
                                 int Hq, int Mq, int q_pos0, float scale, int cand_hi, int keep_k, int tail_lo,
                                 int32_t* idx_out, const fx_kv_out_desc* dst, int64_t dst_stride_layer, void* ws,
                                 size_t ws_bytes, unsigned flags, void* stream)
{
    fx::NvtxRange nvtx_range("fx_kv_retain_per_layer");
    fx_status st = check_kv(kv, "kv");
    if (st != FX_OK) return st;
    if ((st = check_flags(flags)) != FX_OK) return st;
    if (n_layers < 1) return fail(FX_ERR_INVALID_ARG, "n_layers must be >= 1");
    if (!q || !idx_out) return fail(FX_ERR_INVALID_ARG, "q and idx_out must be non-NULL");
    if (cand_hi < 1 || cand_hi > kv->Tcap) return fail(FX_ERR_INVALID_ARG, "need 1 <= cand_hi <= Tcap");
    if (keep_k < 1 || keep_k > cand_hi) return fail(FX_ERR_INVALID_ARG, "need 1 <= keep_k <= cand_hi");
    if (!row_stride_ok(src_stride_layer)) return fail(FX_ERR_INVALID_ARG, "src_stride_layer must be a multiple of 8");
    if ((st = check_heads(Hq, kv->Hkv, Mq)) != FX_OK) return st;
    if (!aligned16(q)) return fail(FX_ERR_INVALID_ARG, "q must be 16-byte aligned");
    if (q_pos0 < -1) return fail(FX_ERR_INVALID_ARG, "q_pos0 must be -1 or >= 0");
    if (!isfinite(scale)) return fail(FX_ERR_INVALID_ARG, "scale must be finite");
    const size_t need = fx_retain_workspace_bytes(kv->B, kv->Hkv, Hq, Mq, kv->Tcap, cand_hi);
    if (need == 0) return fail(FX_ERR_INVALID_ARG, "bad shape");
    if ((st = check_ws(ws, ws_bytes, need)) != FX_OK) return st;
    const size_t fbytes = retain_scoring_bytes(kv->B, kv->Hkv, Hq, Mq, kv->Tcap);
    float* scores = reinterpret_cast<float*>(static_cast<char*>(ws) + fbytes);
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FX_OK) return st;
    const int rows = kv->B * kv->Hkv;
    const size_t q_layer = (size_t)kv->B * Hq * Mq * kHeadDim;
    const size_t layer_scores = (size_t)rows * cand_hi;
    // Every call after the first runs as a programmatic dependent launch when the caller asked for
    // one; the later focal calls read K and lengths that were written before the first call.
    const unsigned pdl = flags & FX_LAUNCH_PDL;
    for (int l0 = 0; l0 < n_layers; l0 += kRetainBatch) {
        const int nb = std::min(kRetainBatch, n_layers - l0);
        fx_kv_desc kb = *kv;
        kb.k = kv->k + (int64_t)l0 * src_stride_layer;
        if (nb > 1 && score_tc_route(ds, &kb, src_stride_layer, nb, q + (size_t)l0 * q_layer, Hq, Mq, q_pos0, scale, 0,
                                     cand_hi, scores, ws, fbytes, pdl != 0, static_cast<cudaStream_t>(stream), &st)) {
            if (st != FX_OK) return st;
        } else for (int l = l0; l < l0 + nb; ++l) {
            fx_kv_desc kl = *kv;
            kl.k = kv->k + (int64_t)l * src_stride_layer;
            kl.v = kv->v + (int64_t)l * src_stride_layer;
            const unsigned ff = l == 0 ? flags : (pdl ? (FX_LAUNCH_PDL | FX_LAUNCH_INPUTS_READY) : 0u);
            st = fx_focal_attn_scores(&kl, q + (size_t)l * q_layer, Hq, Mq, q_pos0, scale, 0, cand_hi, nullptr,
                                      scores + (size_t)(l - l0) * layer_scores, ws, fbytes, ff, stream);
            if (st != FX_OK) return st;
        }
        // the batch's layers' rows are consecutive in both the score rows and idx_out
        st = fx_topk_select(scores, nb * rows, cand_hi, keep_k, nullptr, idx_out + (size_t)l0 * rows * keep_k, pdl, stream);
        if (st != FX_OK) return st;
    }
    return fx_kv_compact(kv, src_stride_layer, idx_out, (int64_t)rows * keep_k, keep_k, tail_lo, dst,
                         dst_stride_layer, n_layers, pdl, stream);
}

// ---------------------------------------------------------------------------------------------
// The dense prefix runs on the tensor cores (its own kernel, partials folded into the verify merge)
// when it fills at least one 128-row by 128-key tile.
bool prefix_on_tensor_cores(bool dense, int P, int Br, int R) { return dense && P >= 128 && (int64_t)Br * R >= 128; }

size_t prefix_ext_bytes(int Br, int Hkv, int R) { return round_up((size_t)Hkv * Br * R * (2 + kHeadDim) * sizeof(float)); }

size_t fx_shared_prefix_workspace_bytes(int Br, int Hkv, int Hq, int Mq, int np, int max_suffix)
{
    if (Br < 1 || Hkv < 1 || Hq < Hkv || Mq < 1 || np < 0 || max_suffix < 0) return 0;
    const int R = (Hq / Hkv) * Mq;
    const Plan pl = make_plan(Br * Hkv, R, np + max_suffix + Mq, sm_count_or_default(), true, np > 0);
    size_t need = make_layout(Br * Hkv, R, pl, 0, true).total;
    if (prefix_on_tensor_cores(true, np, Br, R)) {   // a dense prefix of np rows may take that route
        const Plan pt = make_plan(Br * Hkv, R, max_suffix + Mq, sm_count_or_default(), true, false);
        need = std::max(need, make_layout(Br * Hkv, R, pt, 0, true).total + prefix_ext_bytes(Br, Hkv, R));
    }
    return need;
}

fx_status fx_shared_prefix_decode(const fx_prefix_desc* prefix, const fx_branch_desc* br,
                                  const fx_bf16* q, int Hq, const int32_t* prefix_idx, int kp,
                                  float scale, float* out, void* ws, size_t ws_bytes, unsigned flags,
                                  void* stream)
{
    fx::NvtxRange nvtx_range("fx_shared_prefix_decode");
    if (!prefix || !br) return fail(FX_ERR_INVALID_ARG, "prefix and branches must be non-NULL");
    if (check_flags(flags) != FX_OK) return FX_ERR_INVALID_ARG;
    if (prefix->d != kHeadDim) return fail(FX_ERR_UNSUPPORTED, "head dim %d (only 128 is implemented)", prefix->d);
    if (prefix->P < 0 || prefix->Hkv < 1) return fail(FX_ERR_INVALID_ARG, "need P >= 0 and Hkv >= 1");
    if (!prefix->k || !prefix->v) return fail(FX_ERR_INVALID_ARG, "prefix k/v are NULL");
    if (!aligned16(prefix->k) || !aligned16(prefix->v) || !row_stride_ok(prefix->stride_h) ||
        !row_stride_ok(prefix->stride_t))
        return fail(FX_ERR_INVALID_ARG, "prefix rows must be 16-byte aligned (strides multiples of 8)");
    if (br->Br < 1 || br->Mq < 1) return fail(FX_ERR_INVALID_ARG, "need Br >= 1 and Mq >= 1");
    if (!br->suf_off) return fail(FX_ERR_INVALID_ARG, "suf_off is NULL");
    if (br->suf_rows < 0 || br->max_suffix < 0) return fail(FX_ERR_INVALID_ARG, "need suf_rows, max_suffix >= 0");
    if (br->suf_rows > 0 && (!br->suf_k || !br->suf_v)) return fail(FX_ERR_INVALID_ARG, "suffix k/v are NULL");
    if (!aligned16(br->suf_k) || !aligned16(br->suf_v) || !row_stride_ok(br->suf_stride_h) ||
        !row_stride_ok(br->suf_stride_t))
        return fail(FX_ERR_INVALID_ARG, "suffix rows must be 16-byte aligned (strides multiples of 8)");
    if (!br->draft_k || !br->draft_v || !aligned16(br->draft_k) || !aligned16(br->draft_v) ||
        !row_stride_ok(br->draft_stride_b) || !row_stride_ok(br->draft_stride_i) || !row_stride_ok(br->draft_stride_h))
        return fail(FX_ERR_INVALID_ARG, "draft rows must be non-NULL and 16-byte aligned");
    fx_status st = check_heads(Hq, prefix->Hkv, br->Mq);
    if (st != FX_OK) return st;
    if (!q || !aligned16(q)) return fail(FX_ERR_INVALID_ARG, "q must be non-NULL and 16-byte aligned");
    if (!out) return fail(FX_ERR_INVALID_ARG, "out is NULL");
    if (prefix_idx && kp < 0) return fail(FX_ERR_INVALID_ARG, "kp must be >= 0");
    if (!isfinite(scale)) return fail(FX_ERR_INVALID_ARG, "scale must be finite");
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FX_OK) return st;

    const int Hkv = prefix->Hkv;
    const int pairs = br->Br * Hkv;
    const int G = Hq / Hkv;
    const int R = G * br->Mq;
    const bool tc = prefix_on_tensor_cores(prefix_idx == nullptr, prefix->P, br->Br, R);
    const int np = prefix_idx ? kp : (tc ? 0 : prefix->P);
    const int max_keys = np + br->max_suffix + br->Mq;
    const Plan pl = make_plan(pairs, R, max_keys, ds->sm_count, true, prefix_idx != nullptr);
    const Layout L = make_layout(pairs, R, pl, 0, true);
    const size_t ext_off = L.total;
    if ((st = check_ws(ws, ws_bytes, L.total + (tc ? prefix_ext_bytes(br->Br, Hkv, R) : 0))) != FX_OK) return st;
    if (pairs > 65535 || pl.nsplit > 65535) return fail(FX_ERR_UNSUPPORTED, "grid too large");
    if (tc && (int64_t)br->Br * R / 128 + 1 > 65535) return fail(FX_ERR_UNSUPPORTED, "grid too large");

    char* w = static_cast<char*>(ws);
    AttnParams p;
    memset(&p, 0, sizeof p);
    p.k = prefix->k;
    p.v = prefix->v;
    p.sb = 0;
    p.sh = prefix->stride_h;
    p.st = prefix->stride_t;
    p.B = br->Br;
    p.Hkv = Hkv;
    p.Tcap = prefix->P;
    p.q = q;
    p.Hq = Hq;
    p.G = G;
    p.Mq = br->Mq;
    p.R = R;
    p.q_pos0 = -1;
    p.qscale = log2e_scale(scale);
    p.idx = prefix_idx;
    p.kk = prefix_idx ? kp : 0;
    p.P = prefix->P;
    p.suf_k = br->suf_k;
    p.suf_v = br->suf_v;
    p.suf_sh = br->suf_stride_h;
    p.suf_st = br->suf_stride_t;
    p.suf_off = br->suf_off;
    p.suf_len = br->suf_len;
    p.pre_len = prefix->len;
    p.suf_rows = br->suf_rows;
    p.max_suffix = br->max_suffix;
    p.dr_k = br->draft_k;
    p.dr_v = br->draft_v;
    p.dr_sb = br->draft_stride_b;
    p.dr_si = br->draft_stride_i;
    p.dr_sh = br->draft_stride_h;
    p.nsplit = pl.nsplit;
    p.split_len = pl.split_len;
    p.nrg = pl.nrg;
    p.rb = pl.rb;
    p.stages = pl.stages;
    p.part_m = reinterpret_cast<float*>(w + L.part_m);
    p.part_l = reinterpret_cast<float*>(w + L.part_l);
    p.part_o = reinterpret_cast<float*>(w + L.part_o);
    p.counters = reinterpret_cast<unsigned*>(w + L.counters);
    p.out = out;
    p.err = ds->err;
    bool pdl = (flags & FX_LAUNCH_PDL) != 0;
    p.prefetch = (pdl && (flags & FX_LAUNCH_INPUTS_READY)) ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tc) {
        // the dense prefix of every branch on the tensor cores first; the verify kernel then covers the
        // suffix and draft keys and folds the prefix partials into its merge
        float* ext = reinterpret_cast<float*>(w + ext_off);
        const size_t nrows = (size_t)Hkv * br->Br * R;
        PrefixTcParams t;
        t.pk = reinterpret_cast<const uint16_t*>(prefix->k);
        t.pv = reinterpret_cast<const uint16_t*>(prefix->v);
        t.p_sh = prefix->stride_h;
        t.p_st = prefix->stride_t;
        t.P = prefix->P;
        t.pre_len = prefix->len;
        t.q = reinterpret_cast<const uint16_t*>(q);
        t.Br = br->Br;
        t.Hkv = Hkv;
        t.Hq = Hq;
        t.G = G;
        t.Mq = br->Mq;
        t.R = R;
        t.qscale = p.qscale;
        t.ext_o = ext;   // first: its rows are stored as 16-byte vectors
        t.ext_m = ext + nrows * kHeadDim;
        t.ext_l = t.ext_m + nrows;
        t.err = ds->err;
        cudaError_t e = launch_prefix_tc(t, pdl, s);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core prefix launch");
        p.P = 0;
        p.pre_len = nullptr;
        p.ext_m = t.ext_m;
        p.ext_l = t.ext_l;
        p.ext_o = t.ext_o;
        // the verify kernel's own inputs were all written before this call, so it may read them while
        // the prefix kernel runs (every kernel here triggers only after its own dependency wait)
        pdl = true;
        p.prefetch = 1;
    }
    cudaError_t e = launch_attn_partial(p, kModePrefix, pdl, s);
    if (e != cudaSuccess) return cuda_fail(e, "shared-prefix decode launch");
    return FX_OK;
}

}  // extern "C"

// Tensor maps of one layer's K and V for the streaming decode kernel: [B][Hkv][Tcap][128] bf16 with the
// view's strides, boxes of 16 rows x 64 columns, 128-byte swizzle, rows past Tcap read as zero.
bool fx::encode_kv_tensor_maps(const fx_kv_desc* kv, CUtensorMap* tk, CUtensorMap* tv)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr || kv->Tcap < 1) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)kv->Tcap, (cuuint64_t)kv->Hkv, (cuuint64_t)kv->B};
    const cuuint64_t strides[3] = {(cuuint64_t)kv->stride_t * 2, (cuuint64_t)kv->stride_h * 2, (cuuint64_t)kv->stride_b * 2};
    for (int i = 0; i < 3; ++i)
        if (strides[i] == 0 || (strides[i] & 15u) != 0 || strides[i] >= (1ull << 40)) return false;
    const cuuint32_t box[4] = {64, (cuuint32_t)kSub, 1, 1};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    const void* bases[2] = {kv->k, kv->v};
    CUtensorMap* maps[2] = {tk, tv};
    for (int i = 0; i < 2; ++i) {
        if (fn(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(bases[i]), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool fx::encode_score_maps(const fx_kv_desc* kv, int64_t layer_stride, int layers, const fx_bf16* q, int Hq, int Mq,
                           int n_cols, CUtensorMap* tk, CUtensorMap* tq, int* bcast)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr || kv->Tcap < 1 || layers < 1) return false;
    // a cache shared by every sequence (batch stride 0) is one batch entry of the map
    const bool bc = kv->stride_b == 0;
    const cuuint64_t nb = bc ? 1 : (cuuint64_t)kv->B;
    const cuuint64_t dims[5] = {(cuuint64_t)kHeadDim, (cuuint64_t)kv->Tcap, (cuuint64_t)kv->Hkv, nb,
                                (cuuint64_t)layers};
    const cuuint64_t sb = bc ? (cuuint64_t)kv->stride_h * 2 * (cuuint64_t)kv->Hkv : (cuuint64_t)kv->stride_b * 2;
    // one layer: any stride the encoder accepts (the layer coordinate is always 0)
    const cuuint64_t sl = layers > 1 ? (cuuint64_t)layer_stride * 2 : sb * nb;
    if (layers > 1 && layer_stride <= 0) return false;
    const cuuint64_t strides[4] = {(cuuint64_t)kv->stride_t * 2, (cuuint64_t)kv->stride_h * 2, sb, sl};
    for (int i = 0; i < 4; ++i)
        if (strides[i] == 0 || (strides[i] & 15u) != 0 || strides[i] >= (1ull << 40)) return false;
    const cuuint32_t box[5] = {64, (cuuint32_t)kScoreKeys, 1, 1, 1};
    const cuuint32_t elem[5] = {1, 1, 1, 1, 1};
    if (fn(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(static_cast<const void*>(kv->k)), dims, strides,
           box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    // q as [layers B Hq Mq] rows of 128 bf16 (contiguous); the kernel addresses row starts up to 2^31
    const int64_t qrows = (int64_t)layers * kv->B * Hq * Mq;
    if (qrows >= 0x7fffffff) return false;
    const cuuint64_t qdims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)qrows};
    const cuuint64_t qstrides[1] = {(cuuint64_t)kRowBytes};
    const cuuint32_t qbox[2] = {64, (cuuint32_t)n_cols};
    if (fn(tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(static_cast<const void*>(q)), qdims, qstrides, qbox,
           elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    *bcast = bc ? 1 : 0;
    return true;
}
