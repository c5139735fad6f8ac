// fx_focal_attn_scores_noalloc: the focal call with its scratch in a fixed device array owned by
// the library, for callers that must not allocate device memory themselves.
//
// Some callers cannot allocate: code running while a CUDA graph is being captured (an allocation
// there is either refused or forces a device-wide synchronisation that breaks the capture), hard
// real-time loops that allow no allocator calls after start-up, and hosts that reach the GPU only
// through this C interface and have no allocator of their own.  This entry point takes only the
// inputs and outputs; the split partials and the per-token logits live in g_fx_static_scratch below.
//
// Everything else is the existing fx_focal_attn_scores, called unchanged with that array as its
// workspace.
#include <mutex>

#include "fx_internal.h"

namespace {
constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB
}

// The scratch array.  Every GPU that loads this library holds it until the process exits.  In host
// code its name stands for a host-side shadow, not a device address, so host code obtains the
// device address with cudaGetSymbolAddress (per device) and passes that pointer on.
static __device__ __align__(256) unsigned char g_fx_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
fx_status scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fx::set_error(FX_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return fx::set_error(FX_ERR_CUDA, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fx_static_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fx::set_error(FX_ERR_CUDA, "cudaGetSymbolAddress(static scratch) failed");
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return FX_OK;
}

}  // namespace

extern "C" {

size_t fx_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }

fx_status fx_focal_attn_scores_noalloc(const fx_kv_desc* kv, const fx_bf16* q, int Hq, int Mq, int q_pos0,
                                       float scale, int cand_lo, int cand_hi, float* out, float* scores,
                                       unsigned flags, void* stream)
{
    fx::NvtxRange nvtx_range("fx_focal_attn_scores_noalloc");
    if (!kv) return fx::set_error(FX_ERR_INVALID_ARG, "kv is NULL");
    const size_t need = fx_focal_workspace_bytes(kv->B, kv->Hkv, Hq, Mq, kv->Tcap);
    if (need > kStaticScratchBytes)
        return fx::set_error(FX_ERR_UNSUPPORTED,
                             "this call needs more scratch than the library's fixed 16 MiB array; "
                             "use fx_focal_attn_scores with a workspace of fx_focal_workspace_bytes() bytes");
    void* ws = nullptr;
    fx_status st = scratch_address(&ws);
    if (st != FX_OK) return st;
    return fx_focal_attn_scores(kv, q, Hq, Mq, q_pos0, scale, cand_lo, cand_hi, out, scores, ws,
                                kStaticScratchBytes, flags, stream);
}

}  // extern "C"
