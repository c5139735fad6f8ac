// Split-KV decode attention on CUDA cores for sm_103a.
//
// One CTA = (row group of up to RB query rows, one split of the key sequence, one (b, KV head)).
// The split is walked in tiles of 64 keys.  Each tile's K and V rows (256 bytes each) are copied
// into shared memory with 16-byte cp.async operations -- contiguous rows for the focal mode,
// gathered rows for the sparse and prefix modes -- two tiles in flight at once, so every byte a CTA
// needs is requested before the first one is used.  Rows that must not be read (past the split, or a
// rejected index) are zero-filled by the copy itself.  Each warp then takes 16 keys of the tile: a
// half-warp owns one key per step, lane `sub` holding dims [8*sub, 8*sub+8) (conflict-free 16-byte
// shared loads), the dot products are reduced over the 16 lanes with xor shuffles, and the softmax
// is kept online in base-2 units (q is pre-scaled by scale*log2(e)).  Partial (max, sum,
// unnormalised output) triples per split go to the workspace; the sparse/prefix modes merge them in
// the last-arriving CTA of each (b, h, row group), the focal mode in a separate combine kernel that
// also forms the per-token importance from the stored logits.
//
// Attention and importance follow FastOCR (Methodology: Focal-Guided Pruning): focal layers attend
// over the full cache, the rest over the selected set; FastKV (2.A) for the causal query window;
// HPD-Parsing (parts 2 and 3) for the shared prefix + private suffix + causal draft sequence.
#include <math.h>

#include "fx_internal.h"

namespace fx {
namespace {

constexpr unsigned kFull = 0xffffffffu;

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ void flag(unsigned* err, unsigned bit) { atomicOr(err, bit); }

// Where the rows of one (b, h) key sequence live.  Position pos of the sequence maps to one K row
// and the V row at the same offset from the V base.
template <int MODE>
struct KeySource {
    const uint16_t* kb;   // main cache / prefix base for this (b, h)
    const uint16_t* vb;
    int64_t st;
    int kk;               // gathered positions (sparse idx / prefix idx)
    int tail_lo;          // sparse: tail start token
    int np, L;            // prefix: prefix rows, suffix rows
    const uint16_t* suf_k;
    const uint16_t* suf_v;
    int64_t suf_st;
    const uint16_t* dr_k;
    const uint16_t* dr_v;
    int64_t dr_si;
    bool gathered;        // prefix positions come from s_tok
    int s0;

    // element offset of the row of sequence position `pos` relative to the matching base, and which
    // base to use (0: main, 1: suffix, 2: draft); returns false when the row must not be read.
    __device__ __forceinline__ bool row(int pos, const int* s_tok, const uint16_t*& kp, const uint16_t*& vp) const
    {
        if (MODE == kModeFocal) {
            kp = kb + (int64_t)pos * st;
            vp = vb + (int64_t)pos * st;
            return true;
        }
        if (MODE == kModeSparse) {
            int t;
            if (pos < kk) {
                t = s_tok[pos - s0];
                if (t < 0) return false;
            } else {
                t = tail_lo + (pos - kk);
            }
            kp = kb + (int64_t)t * st;
            vp = vb + (int64_t)t * st;
            return true;
        }
        if (pos < np) {
            int t = pos;
            if (gathered) {
                t = s_tok[pos - s0];
                if (t < 0) return false;
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

template <int MODE, int RB>
__global__ void __launch_bounds__(kThreads) attn_tile_kernel(const AttnParams p)
{
    constexpr int TPC = kTile / (2 * kWarps);   // keys per half-warp per tile (8)
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t* sdata = reinterpret_cast<uint16_t*>(smem_raw);
    int* s_tok = reinterpret_cast<int*>(smem_raw + kStageBytes * kStages);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int hw = lane >> 4;
    const int sub = lane & 15;
    const int rg = blockIdx.x;
    const int split = blockIdx.y;
    const int bh = blockIdx.z;
    const int b = bh / p.Hkv;
    const int h = bh - b * p.Hkv;
    const int r0 = rg * RB;

    // ---- key sequence of this (b, h) ----------------------------------------------------------
    KeySource<MODE> src;
    int n_keys;
    src.kb = p.k + (int64_t)b * p.sb + (int64_t)h * p.sh;
    src.vb = p.v + (int64_t)b * p.sb + (int64_t)h * p.sh;
    src.st = p.st;
    src.kk = p.kk;
    src.tail_lo = p.tail_lo;
    src.gathered = p.idx != nullptr;
    src.np = 0;
    src.L = 0;
    if (MODE == kModeFocal || MODE == kModeSparse) {
        int l = p.len[b];
        if (l < 0 || l > p.Tcap) {
            if (tid == 0) flag(p.err, FX_DEVERR_LEN);
            l = l < 0 ? 0 : p.Tcap;
        }
        n_keys = (MODE == kModeFocal) ? l : p.kk + max(0, l - p.tail_lo);
        src.np = l;   // sparse: valid token range [0, len) for the gathered indices
    } else {
        src.np = p.idx ? p.kk : p.P;
        const int o0 = p.suf_off[b];
        const int o1 = p.suf_off[b + 1];
        int L = 0;
        if (o0 < 0 || o1 < o0 || o1 > p.suf_rows) {
            if (tid == 0) flag(p.err, FX_DEVERR_OFFSETS);
        } else {
            L = o1 - o0;
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
    const int s0 = split * p.split_len;
    const int s1 = min(n_keys, s0 + p.split_len);
    src.s0 = s0;
    const int ntiles = s1 > s0 ? (s1 - s0 + kTile - 1) / kTile : 0;

    // gathered token positions of this split, checked once
    if (MODE != kModeFocal && p.idx != nullptr) {
        const int32_t* irow = p.idx + (int64_t)bh * p.kk;
        const int lim_tok = (MODE == kModeSparse) ? src.np : p.P;
        const int hi = min(s1, p.kk);
        for (int pos = s0 + tid; pos < hi; pos += kThreads) {
            int t = __ldg(irow + pos);
            if (t < 0 || t >= lim_tok) {
                flag(p.err, FX_DEVERR_INDEX);
                t = -1;
            }
            s_tok[pos - s0] = t;
        }
        __syncthreads();
    }

    // ---- tile loader: thread copies 16-byte chunk `sub` of rows (tid >> 4) + 8u, K and V ----------
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sdata);
    auto issue = [&](int tile, int stage) {
        const int base = s0 + tile * kTile;
#pragma unroll
        for (int u = 0; u < kTile / 8; ++u) {
            const int r = (tid >> 4) + 8 * u;
            const int pos = base + r;
            const uint16_t* kp = src.kb;
            const uint16_t* vp = src.vb;
            const bool ok = pos < s1 && src.row(pos, s_tok, kp, vp);
            const uint32_t dk = sbase + (uint32_t)(((stage * 2 + 0) * kTile + r) * kRowBytes + sub * 16);
            const uint32_t dv = sbase + (uint32_t)(((stage * 2 + 1) * kTile + r) * kRowBytes + sub * 16);
            cp_async16(dk, ok ? (const void*)(kp + sub * 8) : (const void*)src.kb, ok ? 16 : 0);
            cp_async16(dv, ok ? (const void*)(vp + sub * 8) : (const void*)src.vb, ok ? 16 : 0);
        }
        cp_async_commit();
    };

    // ---- query rows: lane `sub` holds dims [8*sub, 8*sub+8) of each row ------------------------
    float qf[RB][8];
    int lim[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int row = r0 + r;
        if (row < p.R) {
            const int gi = row / p.Mq;
            const int i = row - gi * p.Mq;
            const uint16_t* qp = p.q + ((((int64_t)b * p.Hq + h * p.G + gi) * p.Mq + i) << 7) + sub * 8;
            const uint4 w = *reinterpret_cast<const uint4*>(qp);
            unpack8(w, qf[r]);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[r][e] *= p.qscale;
            if (MODE == kModeFocal)
                lim[r] = p.q_pos0 >= 0 ? p.q_pos0 + i : 0x7fffffff;
            else if (MODE == kModePrefix)
                lim[r] = src.np + src.L + i;   // draft row j is visible iff j <= i
            else
                lim[r] = 0x7fffffff;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[r][e] = 0.f;
            lim[r] = -1;   // padding row: sees nothing
        }
    }

    float m[RB], l[RB], o[RB][8];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][e] = 0.f;
    }

    if (ntiles > 0) issue(0, 0);
    if (ntiles > 1) issue(1, 1);

    for (int tile = 0; tile < ntiles; ++tile) {
        const int stage = tile & 1;
        if (tile + 1 < ntiles)
            cp_async_wait_all_but_one();
        else
            cp_async_wait_all();
        __syncthreads();

        const int base = s0 + tile * kTile;
        const uint16_t* sK = sdata + (size_t)(stage * 2 + 0) * kTile * kHeadDim;
        const uint16_t* sV = sdata + (size_t)(stage * 2 + 1) * kTile * kHeadDim;

        float lg[TPC][RB];
        bool valid[TPC];
        int pos[TPC];
#pragma unroll
        for (int i = 0; i < TPC; ++i) {
            const int row = warp * (2 * TPC) + 2 * i + hw;
            pos[i] = base + row;
            bool ok = pos[i] < s1;
            if (MODE == kModeSparse && ok && pos[i] < p.kk) ok = s_tok[pos[i] - s0] >= 0;
            if (MODE == kModePrefix && ok && src.gathered && pos[i] < src.np) ok = s_tok[pos[i] - s0] >= 0;
            valid[i] = ok;
            float kf[8];
            unpack8(*reinterpret_cast<const uint4*>(sK + row * kHeadDim + sub * 8), kf);
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(qf[r][e], kf[e], s);
                s += __shfl_xor_sync(kFull, s, 8);
                s += __shfl_xor_sync(kFull, s, 4);
                s += __shfl_xor_sync(kFull, s, 2);
                s += __shfl_xor_sync(kFull, s, 1);
                lg[i][r] = (ok && pos[i] <= lim[r]) ? s : -INFINITY;
            }
        }

        if (MODE == kModeFocal && p.logits != nullptr) {
            const int pp = base + warp * (2 * TPC) + 2 * sub + hw;
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                if (r0 + r < p.R) {
                    float mine = lg[0][r];
#pragma unroll
                    for (int i = 1; i < TPC; ++i)
                        if (sub == i) mine = lg[i][r];
                    if (sub < TPC && pp < s1) p.logits[(int64_t)(bh * p.R + r0 + r) * p.Tcap + pp] = mine;
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
            const int row = warp * (2 * TPC) + 2 * i + hw;
            float vf[8];
            unpack8(*reinterpret_cast<const uint4*>(sV + row * kHeadDim + sub * 8), vf);
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int e = 0; e < 8; ++e) o[r][e] = fmaf(lg[i][r], vf[e], o[r][e]);
        }
        __syncthreads();                       // every warp is done with this stage
        if (tile + 2 < ntiles) issue(tile + 2, stage);
    }

    // the two half-warps hold the same dims for different keys
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        l[r] += __shfl_xor_sync(kFull, l[r], 16);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][e] += __shfl_xor_sync(kFull, o[r][e], 16);
    }

    // ---- combine the warps of this CTA into one partial per row (tile buffers are free now) ----
    __shared__ float sm_m[kWarps][RB];
    __shared__ float sm_l[kWarps][RB];
    float* sm_o = reinterpret_cast<float*>(smem_raw);   // [kWarps][RB][128]
    if (lane < 16) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float4* dst = reinterpret_cast<float4*>(sm_o + (warp * RB + r) * kHeadDim + sub * 8);
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
            O = fmaf(sm_o[(w * RB + r) * kHeadDim + tid], sc, O);
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

template <int MODE, int RB>
cudaError_t launch_one(const AttnParams& p, size_t smem, cudaStream_t s)
{
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(attn_tile_kernel<MODE, RB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)attn_smem_bytes(kMaxSplitTokens));
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    dim3 grid(p.nrg, p.nsplit, p.B * p.Hkv);
    attn_tile_kernel<MODE, RB><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const AttnParams& p, int rb, cudaStream_t s)
{
    const size_t smem = attn_smem_bytes((MODE != kModeFocal && p.idx != nullptr) ? p.split_len : 0);
    switch (rb) {
    case 1: return launch_one<MODE, 1>(p, smem, s);
    case 2: return launch_one<MODE, 2>(p, smem, s);
    case 4: return launch_one<MODE, 4>(p, smem, s);
    default: return launch_one<MODE, 8>(p, smem, s);
    }
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
