// Split-KV decode attention on CUDA cores for sm_103a.
//
// One CTA = (row group of up to RB query rows, one split of the key sequence, one (b, KV head)).
// Each warp walks chunks of 2*TPC keys; within a chunk a half-warp owns one key per step: lane
// `sub` (0..15) loads 16 bytes (8 bf16 of the 128-wide row) of K and of V with one vectorised
// load each, so a warp instruction moves two full 256-byte rows.  Logits are reduced over the 16
// lanes with xor shuffles, the softmax is kept online in base-2 units (q is pre-scaled by
// scale*log2(e)), and V is accumulated straight from registers: K/V bytes are touched exactly once
// and never staged.  Partial (max, sum, unnormalised output) triples per split go to the
// workspace; the sparse/prefix modes merge them in the last-arriving CTA of each (b, h, row group),
// the focal mode in a separate combine kernel that also forms the per-token importance.
//
// Attention and importance follow FastOCR (Methodology: Focal-Guided Pruning): focal layers attend
// over the full cache, the rest over the selected set; FastKV (2.A) for the causal query window.
#include <math.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint4 ld_stream16(const uint16_t* ptr)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(ptr));
    return r;
}

__device__ __forceinline__ void unpack8(const uint4& w, float f[8])
{
    // bf16 -> fp32 is a 16-bit left shift of the pattern; element 2i is the low half of word i.
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
    f[4] = __uint_as_float(w.z << 16);
    f[5] = __uint_as_float(w.z & 0xffff0000u);
    f[6] = __uint_as_float(w.w << 16);
    f[7] = __uint_as_float(w.w & 0xffff0000u);
}

__device__ __forceinline__ void flag(unsigned* err, unsigned bit) { atomicOr(err, bit); }

template <int MODE, int RB>
__global__ void __launch_bounds__(kThreads) attn_partial_kernel(const AttnParams p)
{
    constexpr int TPC = (RB >= 8) ? 4 : 8;  // keys per half-warp per chunk
    constexpr int CH = 2 * TPC;             // keys per warp per chunk

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int hw = lane >> 4;
    const int sub = lane & 15;
    const int rg = blockIdx.x;
    const int split = blockIdx.y;
    const int bh = blockIdx.z;
    const int b = bh / p.Hkv;
    const int h = bh - b * p.Hkv;
    const int r0 = rg * RB;

    // ---- key sequence of this (b, h) ----------------------------------------------------------
    int n_keys;
    int lenb = 0, np = 0, L = 0, soff = 0;
    if (MODE == kModeFocal || MODE == kModeSparse) {
        int l = p.len[b];
        if (l < 0 || l > p.Tcap) {
            if (threadIdx.x == 0) flag(p.err, FX_DEVERR_LEN);
            l = l < 0 ? 0 : p.Tcap;
        }
        lenb = l;
        n_keys = (MODE == kModeFocal) ? lenb : p.kk + max(0, lenb - p.tail_lo);
    } else {
        np = p.idx ? p.kk : p.P;
        const int o0 = p.suf_off[b];
        const int o1 = p.suf_off[b + 1];
        if (o0 < 0 || o1 < o0 || o1 > p.suf_rows) {
            if (threadIdx.x == 0) flag(p.err, FX_DEVERR_OFFSETS);
            L = 0;
        } else {
            L = o1 - o0;
            if (L > p.max_suffix) {
                if (threadIdx.x == 0) flag(p.err, FX_DEVERR_OFFSETS);
                L = p.max_suffix;
            }
        }
        soff = o0;
        n_keys = np + L + p.Mq;
    }
    const int s0 = split * p.split_len;
    const int s1 = min(n_keys, s0 + p.split_len);

    // ---- query rows: lane `sub` holds dims [8*sub, 8*sub+8) of each row ------------------------
    float qf[RB][8];
    int lim[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int row = r0 + r;
        if (row < p.R) {
            const int gi = row / p.Mq;
            const int i = row - gi * p.Mq;
            const uint16_t* qp =
                p.q + ((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + sub * 8;
            const uint4 w = *reinterpret_cast<const uint4*>(qp);
            unpack8(w, qf[r]);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[r][e] *= p.qscale;
            if (MODE == kModeFocal)
                lim[r] = p.q_pos0 >= 0 ? p.q_pos0 + i : 0x7fffffff;
            else if (MODE == kModePrefix)
                lim[r] = np + L + i;   // draft row j is visible iff j <= i
            else
                lim[r] = 0x7fffffff;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[r][e] = 0.f;
            lim[r] = -1;                // padding row: sees nothing
        }
    }

    const uint16_t* kb = p.k + (int64_t)b * p.sb + (int64_t)h * p.sh;
    const uint16_t* vb = p.v + (int64_t)b * p.sb + (int64_t)h * p.sh;
    const int32_t* idxrow = p.idx ? p.idx + (int64_t)bh * p.kk : nullptr;

    float m[RB], l[RB], o[RB][8];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][e] = 0.f;
    }

    for (int cbase = s0 + warp * CH; cbase < s1; cbase += kWarps * CH) {
        // gathered token positions of this chunk, one per lane, broadcast below
        int myidx = 0;
        if (MODE != kModeFocal && idxrow != nullptr) {
            const int pp = cbase + lane;
            if (lane < CH && pp < s1 && pp < p.kk) myidx = __ldg(idxrow + pp);
        }

        uint4 kr[TPC], vr[TPC];
        bool valid[TPC];
        int pos[TPC];
#pragma unroll
        for (int i = 0; i < TPC; ++i) {
            pos[i] = cbase + 2 * i + hw;
            const int tsrc = __shfl_sync(kFull, myidx, 2 * i + hw);
            bool ok = pos[i] < s1;
            const uint16_t* kp = kb;
            const uint16_t* vp = vb;
            if (MODE == kModeFocal) {
                kp = kb + (int64_t)pos[i] * p.st;
                vp = vb + (int64_t)pos[i] * p.st;
            } else if (MODE == kModeSparse) {
                int t;
                if (pos[i] < p.kk) {
                    t = tsrc;
                    if (ok && (t < 0 || t >= lenb)) {
                        flag(p.err, FX_DEVERR_INDEX);
                        ok = false;
                    }
                } else {
                    t = p.tail_lo + (pos[i] - p.kk);
                }
                kp = kb + (int64_t)t * p.st;
                vp = vb + (int64_t)t * p.st;
            } else {
                if (pos[i] < np) {
                    int t = idxrow ? tsrc : pos[i];
                    if (ok && idxrow && (t < 0 || t >= p.P)) {
                        flag(p.err, FX_DEVERR_INDEX);
                        ok = false;
                    }
                    kp = kb + (int64_t)t * p.st;
                    vp = vb + (int64_t)t * p.st;
                } else if (pos[i] < np + L) {
                    const int64_t t = soff + (pos[i] - np);
                    kp = p.suf_k + (int64_t)h * p.suf_sh + t * p.suf_st;
                    vp = p.suf_v + (int64_t)h * p.suf_sh + t * p.suf_st;
                } else {
                    const int64_t j = pos[i] - np - L;
                    kp = p.dr_k + (int64_t)b * p.dr_sb + j * p.dr_si + (int64_t)h * p.dr_sh;
                    vp = p.dr_v + (int64_t)b * p.dr_sb + j * p.dr_si + (int64_t)h * p.dr_sh;
                }
            }
            valid[i] = ok;
            if (ok) {
                kr[i] = ld_stream16(kp + sub * 8);
                vr[i] = ld_stream16(vp + sub * 8);
            } else {
                kr[i] = make_uint4(0u, 0u, 0u, 0u);
                vr[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }

        // logits (base 2), reduced over the 16 lanes of each half-warp
        float lg[TPC][RB];
#pragma unroll
        for (int i = 0; i < TPC; ++i) {
            float kf[8];
            unpack8(kr[i], kf);
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(qf[r][e], kf[e], s);
                s += __shfl_xor_sync(kFull, s, 8);
                s += __shfl_xor_sync(kFull, s, 4);
                s += __shfl_xor_sync(kFull, s, 2);
                s += __shfl_xor_sync(kFull, s, 1);
                lg[i][r] = (valid[i] && pos[i] <= lim[r]) ? s : -INFINITY;
            }
        }

        if (MODE == kModeFocal && p.logits != nullptr) {
            const int pp = cbase + 2 * sub + hw;
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                if (r0 + r < p.R) {
                    float mine = lg[0][r];
#pragma unroll
                    for (int i = 1; i < TPC; ++i)
                        if (sub == i) mine = lg[i][r];
                    if (sub < TPC && pp < s1)
                        p.logits[(int64_t)(bh * p.R + r0 + r) * p.Tcap + pp] = mine;
                }
            }
        }

        // online softmax update
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float cm = lg[0][r];
#pragma unroll
            for (int i = 1; i < TPC; ++i) cm = fmaxf(cm, lg[i][r]);
            cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, 16));
            const float mn = fmaxf(m[r], cm);
            const float ms = (mn == -INFINITY) ? 0.f : mn;
            const float alpha = exp2f(m[r] - ms);
            l[r] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[r][e] *= alpha;
            m[r] = mn;
#pragma unroll
            for (int i = 0; i < TPC; ++i) {
                lg[i][r] = exp2f(lg[i][r] - ms);
                l[r] += lg[i][r];
            }
        }
#pragma unroll
        for (int i = 0; i < TPC; ++i) {
            float vf[8];
            unpack8(vr[i], vf);
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int e = 0; e < 8; ++e) o[r][e] = fmaf(lg[i][r], vf[e], o[r][e]);
        }
    }

    // the two half-warps hold the same dims for different keys
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        l[r] += __shfl_xor_sync(kFull, l[r], 16);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][e] += __shfl_xor_sync(kFull, o[r][e], 16);
    }

    // ---- combine the warps of this CTA into one partial per row -------------------------------
    __shared__ float sm_m[kWarps][RB];
    __shared__ float sm_l[kWarps][RB];
    __shared__ __align__(16) float sm_o[kWarps][RB][kHeadDim];
    if (lane < 16) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float4* dst = reinterpret_cast<float4*>(&sm_o[warp][r][sub * 8]);
            dst[0] = make_float4(o[r][0], o[r][1], o[r][2], o[r][3]);
            dst[1] = make_float4(o[r][4], o[r][5], o[r][6], o[r][7]);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            sm_m[warp][r] = m[r];
            sm_l[warp][r] = l[r];
        }
    }
    __syncthreads();

    const int tid = threadIdx.x;  // == output dim
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int row = r0 + r;
        if (row >= p.R) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][r]);
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float sc = exp2f(sm_m[w][r] - Ms);
            Ls = fmaf(sm_l[w][r], sc, Ls);
            O = fmaf(sm_o[w][r][tid], sc, O);
        }
        const int64_t pi = (int64_t)(bh * p.R + row) * p.nsplit + split;
        p.part_o[pi * kHeadDim + tid] = O;
        if (tid == 0) {
            p.part_m[pi] = M;
            p.part_l[pi] = Ls;
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
    for (int r = 0; r < RB; ++r) {
        const int row = r0 + r;
        if (row >= p.R) continue;
        const int64_t base = (int64_t)(bh * p.R + row) * p.nsplit;
        float M = -INFINITY;
        for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, __ldcg(p.part_m + base + s));
        const float Ms = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f, O = 0.f;
        for (int s = 0; s < p.nsplit; ++s) {
            const float sc = exp2f(__ldcg(p.part_m + base + s) - Ms);
            Ls = fmaf(__ldcg(p.part_l + base + s), sc, Ls);
            O = fmaf(__ldcg(p.part_o + (base + s) * kHeadDim + tid), sc, O);
        }
        const int gi = row / p.Mq;
        const int i = row - gi * p.Mq;
        p.out[((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + tid] = Ls > 0.f ? O / Ls : 0.f;
    }
    if (tid == 0) p.counters[bh * p.nrg + rg] = 0u;
}

// Focal combine: merge split partials into the output rows and form the importance scores
//   s_j = sum_r exp2(t_rj - M_r) / Z_r   over the group's rows r, for cand_lo <= j < cand_hi.
__global__ void __launch_bounds__(256) focal_combine_kernel(const FocalCombineParams p)
{
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
        for (int s = 0; s < p.nsplit; ++s) Z = fmaf(p.part_l[base + s], exp2f(p.part_m[base + s] - Ms), Z);
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
                O = fmaf(p.part_o[(base + s) * kHeadDim + c], exp2f(p.part_m[base + s] - sM[r]), O);
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
                    s = fmaf(exp2f(__ldcs(lrow + (int64_t)r * p.Tcap + j) - sM[r]), sInvZ[r], s);
            }
            srow[jj] = s;
        }
    }
}

template <int MODE>
cudaError_t launch_mode(const AttnParams& p, int rb, cudaStream_t s)
{
    dim3 grid(p.nrg, p.nsplit, p.B * p.Hkv);
    switch (rb) {
    case 1: attn_partial_kernel<MODE, 1><<<grid, kThreads, 0, s>>>(p); break;
    case 2: attn_partial_kernel<MODE, 2><<<grid, kThreads, 0, s>>>(p); break;
    case 4: attn_partial_kernel<MODE, 4><<<grid, kThreads, 0, s>>>(p); break;
    default: attn_partial_kernel<MODE, 8><<<grid, kThreads, 0, s>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_partial(const AttnParams& p, int mode, int rb, cudaStream_t s)
{
    if (mode == kModeFocal) return launch_mode<kModeFocal>(p, rb, s);
    if (mode == kModeSparse) return launch_mode<kModeSparse>(p, rb, s);
    return launch_mode<kModePrefix>(p, rb, s);
}

cudaError_t launch_focal_combine(const FocalCombineParams& p, cudaStream_t s)
{
    const int ncand = p.scores ? (p.cand_hi - p.cand_lo) : 0;
    int gx = (ncand + 1023) / 1024;
    if (gx < 1) gx = 1;
    if (gx > 256) gx = 256;
    dim3 grid(gx, p.B * p.Hkv);
    focal_combine_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace fx
