// Device helpers shared by the attention kernels (mma.sync fragments, ldmatrix, cp.async, cluster
// stores and mbarriers).  Inline PTX for sm_103a; every function is internal to the including unit.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---- PTX wrappers -------------------------------------------------------------------------------
__device__ __forceinline__ float fast_exp2(float x)   // hardware 2^x (relative error about 2^-22)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// all of this thread's commit groups but the newest WS-1 have completed
template <int WS>
__device__ __forceinline__ void cp_async_wait_stages()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(WS - 1) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all_groups() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// Byte offset of 16-byte chunk `chunk` (0..15) of row `row` in a staged K or V sub-tile: rows are
// 256 bytes apart and the chunk index is XORed with (row % 8), so the 8 rows an ldmatrix reads at one
// column fall on 8 distinct bank groups without padding.
__device__ __forceinline__ uint32_t kv_off(int row, int chunk)
{
    return (uint32_t)(row * kKvPitch + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D (fp32)
__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// transpose of an 8x8 b16 matrix held one 32-bit pair per lane (row lane/4, columns 2*(lane%4) + 0, 1)
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), for a pair of values
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
    hi = *reinterpret_cast<uint32_t*>(&hv);
    lo = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
}

__device__ __forceinline__ void flag(unsigned* err, unsigned bit) { atomicOr(err, bit); }

__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// asynchronous stores into another CTA's shared memory that complete bytes on that CTA's mbarrier
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr), "f"(v),
                 "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_for_cluster(uint64_t* bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, unsigned parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---- CTA-local mbarriers (producer / consumer rings) ------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// plain arrival (release at CTA scope): the arriving thread's earlier shared-memory accesses are ordered
// before a thread that observes the phase completing
__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// arrival that fires once every cp.async this thread issued before it has landed (the pending count is
// raised now and lowered by that asynchronous arrival, so it needs no slot in the initial count)
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Waits for the phase of `parity` to complete, giving up after `limit` polls (then sets
// FX_DEVERR_TIMEOUT and returns false: the caller's results are invalid but nothing hangs).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity, unsigned* err, unsigned limit)
{
    unsigned spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (++spins >= limit) {
            atomicOr(err, FX_DEVERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

}  // namespace
}  // namespace fx
