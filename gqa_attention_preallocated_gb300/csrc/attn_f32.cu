// Generic GQA attention: fp32 storage (d <= 256, d % 4 == 0), and bf16
// storage of a head dimension other than the 128 the TMA / tensor-core
// kernels take (d <= 256, d % 8 == 0).  Values are widened to fp32 as they
// are staged in shared memory; scores, softmax and the output accumulate in
// fp32; a bf16 cache takes bf16 queries and writes bf16 outputs (rounded to
// nearest even).
//
// Semantics ("Implement grouped-query attention over a preallocated KV
// cache...", "A strong answer", gqa_attention): query (b, h, t) with
// t < n_new[b] sits at position prior[b] + t (prior = lens - n_new) and
// attends to keys 0 .. prior[b] + t of KV head h / G with softmax scale
// 1/sqrt(d); padded queries give 0.  The mask is index arithmetic ("Write
// the causal mask for a decode step...", bottom-right rule j <= i + S - T).
//
// One CTA serves a block of 16 query rows r = g*T + t of one KV head, so the
// K/V tile it stages in shared memory is read once for up to 16 query rows
// (all G heads of the group when G*T <= 16).  Each warp owns 4 rows; lane j
// scores keys j and j + 32 of the 64-key tile, the warp keeps a running max
// and sum (online softmax) and lane e accumulates output dims e, e+32, ...
// Masked keys are skipped outright, so stale or NaN slots past lens never
// enter.
//
// Sliding window and ring storage ("Write the causal mask for a decode
// step...", "A strong answer", last paragraph): with a window W the query at
// position p sees keys p - W < a <= p, and in a ring cache key a is read from
// slot a mod max_len; keys are chosen by position, never by slot.  Tree
// verify ("What interviewers probe next", tree-based speculative decoding):
// a query sees the chunk's tokens on its own path to the root only.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kRows = 16;
constexpr int kKeys = 64;  // key tile: two keys a lane
constexpr int kWarps = 4;
constexpr int kMaxD = 256;

__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_out(float* dst, float x) { *dst = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* dst, float x) { *dst = __float2bfloat16_rn(x); }

// 16 E4M3 codes -> 16 values times the head's scale (E4M3 -> f16 is exact).
__device__ __forceinline__ void widen_e4m3x16(const uint8_t* src, float sc, float (&f)[16]) {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t lo, hi;
        ptx::e4m3x4_to_f16x2x2(u[i], lo, hi);  // bytes 0, 1 -> lo; 2, 3 -> hi (low half first)
        __half2 hl, hh;
        memcpy(&hl, &lo, 4);
        memcpy(&hh, &hi, 4);
        const float2 a = __half22float2(hl), b = __half22float2(hh);
        f[4 * i] = a.x * sc;
        f[4 * i + 1] = a.y * sc;
        f[4 * i + 2] = b.x * sc;
        f[4 * i + 3] = b.y * sc;
    }
}

// 16 stored bytes (4 fp32, 8 bf16 or 16 E4M3 values) into fp32 shared memory.
__device__ __forceinline__ void stage16(float* dst, const uint8_t* src, float sc) {
    float f[16];
    widen_e4m3x16(src, sc, f);
#pragma unroll
    for (int i = 0; i < 4; ++i) reinterpret_cast<float4*>(dst)[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
}
__device__ __forceinline__ void stage16(float* dst, const float* src) {
    *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(src);
}
__device__ __forceinline__ void stage16(float* dst, const __nv_bfloat16* src) {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // bf16 -> fp32 is exact: the bits move up 16
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
    reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ void stage16(float* dst, const float* src, float) { stage16(dst, src); }
__device__ __forceinline__ void stage16(float* dst, const __nv_bfloat16* src, float) { stage16(dst, src); }

// The same into a row of any alignment (one value a store).
__device__ __forceinline__ void stage16_rows(float* dst, const uint8_t* src, float sc) {
    float f[16];
    widen_e4m3x16(src, sc, f);
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[i] = f[i];
}
__device__ __forceinline__ void stage16_rows(float* dst, const float* src, float) {
    const float4 v = *reinterpret_cast<const float4*>(src);
    dst[0] = v.x;
    dst[1] = v.y;
    dst[2] = v.z;
    dst[3] = v.w;
}
__device__ __forceinline__ void stage16_rows(float* dst, const __nv_bfloat16* src, float) {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dst[2 * i] = __uint_as_float(u[i] << 16);
        dst[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// SE: the stored type (float, bf16, or E4M3 codes as uint8_t); IE: the type
// of the queries and outputs.
template <typename SE, typename IE>
__global__ void __launch_bounds__(kWarps * 32) attn_f32_kernel(const __grid_constant__ F32Params p) {
    constexpr int kVec = 16 / static_cast<int>(sizeof(SE));  // values per 16-byte load
    constexpr bool kF8 = std::is_same<SE, uint8_t>::value;
    const IE* qg = static_cast<const IE*>(p.q);
    const SE* kg = static_cast<const SE*>(p.k_cache);
    const SE* vg = static_cast<const SE*>(p.v_cache);
    IE* og = static_cast<IE*>(p.out);
    extern __shared__ float4 smem4[];
    float* sq = reinterpret_cast<float*>(smem4);  // [kRows][d]
    // K rows are d + 1 floats apart: lane j reads key j's row in the score
    // loop, and an odd stride puts the 32 lanes in 32 different banks.
    const int dk = p.d + 1;
    float* sk = sq + kRows * p.d;                 // [kKeys][d + 1]
    float* sv = sk + kKeys * dk;                  // [kKeys][d] (16-byte aligned: 80 d + 64 floats in)

    const int split = blockIdx.x % p.splits, rb = blockIdx.x / p.splits;
    const int b = blockIdx.z, kvh = blockIdx.y, row0 = rb * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = p.d, T = p.T;
    const int prior = p.prior[b], nn = p.n_new[b];
    const float ksc = kF8 ? p.kscale[kvh] : 1.f, vsc = kF8 ? p.vscale[kvh] : 1.f;  // FP8 code scales

    // Row limits (largest visible key; -1 = padded / missing row), the keys'
    // extent and, with a window, the first key any row of the block sees.
    int lim[4];
    int extent = 0, first = 0x7fffffff;
    for (int i = 0; i < kRows; ++i) {
        const int r = row0 + i;
        int l = -1;
        if (r < p.R && (r % T) < nn) l = prior + (r % T);
        if (l + 1 > extent) extent = l + 1;
        if (l >= 0) first = min(first, p.window > 0 ? max(0, l - p.window + 1) : 0);
        if ((i & 3) == warp) lim[i >> 2] = l;
    }
    if (extent == 0) first = 0;
    // This CTA's share of the key range: a contiguous run of 64-key tiles.
    int kbeg = first, kend = extent;
    if (p.splits > 1) {
        const long long ntile = (extent - first + kKeys - 1) / kKeys;
        kbeg = first + static_cast<int>(split * ntile / p.splits) * kKeys;
        kend = min(extent, first + static_cast<int>((split + 1) * ntile / p.splits) * kKeys);
    }

    // Stage the block's query rows.
    for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
        const int i = idx / d, e = idx % d, r = row0 + i;
        float v = 0.f;
        if (r < p.R) {
            const int g = r / T, t = r % T;
            v = widen(qg[((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * T + t) * d + e]);
        }
        sq[idx] = v;
    }

    float m[4], l[4], o[4][kMaxD / 32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) o[i][c] = 0.f;
    }

    for (int k0 = kbeg; k0 < kend; k0 += kKeys) {
        __syncthreads();
        const int nk = min(kKeys, kend - k0);
        for (int idx = threadIdx.x; idx < kKeys * d / kVec; idx += blockDim.x) {
            const int j = (idx * kVec) / d;
            bool live = false;
            size_t off = 0;
            if (j < nk) {
                const int a = k0 + j;  // key position
                bool bad = false;
                const int row = phys_row(p.pg, p.ring, p.Hkv, p.max_len, b, kvh, a, &bad);
                live = !bad;  // a bad block-table entry reads as zeros
                off = static_cast<size_t>(row) * d + static_cast<size_t>(idx * kVec - j * d);
            }
            float* kdst = sk + j * dk + (idx * kVec - j * d);
            if (live) {
                stage16_rows(kdst, kg + off, ksc);
                stage16(sv + idx * kVec, vg + off, vsc);
            } else {
#pragma unroll
                for (int i = 0; i < kVec; ++i) kdst[i] = sv[idx * kVec + i] = 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int li = lim[i];
            const int lo = p.window > 0 ? li - p.window : -1;  // keys <= lo are outside the window
            if (li < k0 || lo >= k0 + nk - 1) continue;  // row sees nothing in this tile (warp-uniform)
            const float* qr = sq + (warp + 4 * i) * d;
            // lane scores keys k0 + lane and k0 + lane + 32
            float sc[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int jj = lane + 32 * h, key = k0 + jj;
                sc[h] = -INFINITY;
                // (key - prior <= li - prior < T <= 64 whenever the bit is read)
                const bool on_path =
                    !p.tree || key < prior || key > li || ((p.anc[b * T + (li - prior)] >> (key - prior)) & 1ull);
                if (jj < nk && key <= li && key > lo && on_path) {
                    // four independent partial sums (d is a multiple of 4)
                    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                    const float* kr = sk + jj * dk;
                    for (int e = 0; e < d; e += 4) {
                        a0 = fmaf(qr[e], kr[e], a0);
                        a1 = fmaf(qr[e + 1], kr[e + 1], a1);
                        a2 = fmaf(qr[e + 2], kr[e + 2], a2);
                        a3 = fmaf(qr[e + 3], kr[e + 3], a3);
                    }
                    sc[h] = ((a0 + a1) + (a2 + a3)) * p.scale;
                }
            }
            float tmax = fmaxf(sc[0], sc[1]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            // A draft tree can leave a row no visible key in a tile (and none
            // before it): then nothing changes.
            const float mnew = fmaxf(m[i], tmax);
            const float alpha = (mnew == -INFINITY) ? 1.f : expf(m[i] - mnew);
            const float p0 = (sc[0] == -INFINITY) ? 0.f : expf(sc[0] - mnew);
            const float p1 = (sc[1] == -INFINITY) ? 0.f : expf(sc[1] - mnew);
            float psum = p0 + p1;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l[i] = l[i] * alpha + psum;
            m[i] = mnew;
#pragma unroll
            for (int c = 0; c < kMaxD / 32; ++c) o[i][c] *= alpha;
            const int jmax = min(nk, li - k0 + 1);
            for (int j = max(0, lo - k0 + 1); j < jmax; ++j) {
                const float pb = __shfl_sync(0xffffffffu, j < 32 ? p0 : p1, j & 31);
                const float* vr = sv + j * d;
#pragma unroll
                for (int c = 0; c < kMaxD / 32; ++c) {
                    const int e = lane + 32 * c;
                    if (e < d) o[i][c] = fmaf(pb, vr[e], o[i][c]);
                }
            }
        }
    }

    if (p.splits == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = row0 + warp + 4 * i;
            if (r >= p.R) continue;
            const int g = r / T, t = r % T;
            IE* dst = og + ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * T + t) * d;
            const float inv = (lim[i] >= 0 && l[i] > 0.f) ? 1.f / l[i] : 0.f;
#pragma unroll
            for (int c = 0; c < kMaxD / 32; ++c) {
                const int e = lane + 32 * c;
                if (e < d) store_out(dst + e, (lim[i] >= 0) ? o[i][c] * inv : 0.f);
            }
        }
        return;
    }

    // Split key range: leave this CTA's (O, m, l) per row, then the last CTA
    // of the unit to arrive merges every split's state (no waiting):
    // o = sum_s e^(m_s - M) O_s / sum_s e^(m_s - M) l_s, with M = max_s m_s.
    const int unit = (b * p.Hkv + kvh) * (gridDim.x / p.splits) + rb;
    const size_t stride = static_cast<size_t>(d) + 2;
    float* part = p.partials + (static_cast<size_t>(unit) * p.splits + split) * kRows * stride;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float* pr = part + (warp + 4 * i) * stride;
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) {
            const int e = lane + 32 * c;
            if (e < d) pr[e] = o[i][c];
        }
        if (lane == 0) {
            pr[d] = m[i];
            pr[d + 1] = l[i];
        }
    }
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.counters + unit, 1) == p.splits - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* ups = p.partials + static_cast<size_t>(unit) * p.splits * kRows * stride;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int rr = warp + 4 * i, r = row0 + rr;
        if (r >= p.R) continue;
        float M = -INFINITY;
        for (int sp = 0; sp < p.splits; ++sp) M = fmaxf(M, __ldcg(ups + (sp * kRows + rr) * stride + d));
        float L = 0.f, acc[kMaxD / 32];
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) acc[c] = 0.f;
        for (int sp = 0; sp < p.splits; ++sp) {
            const float* pr = ups + (sp * kRows + rr) * stride;
            const float ms = __ldcg(pr + d);
            const float w = (ms == -INFINITY) ? 0.f : expf(ms - M);
            L += w * __ldcg(pr + d + 1);
#pragma unroll
            for (int c = 0; c < kMaxD / 32; ++c) {
                const int e = lane + 32 * c;
                if (e < d) acc[c] += w * __ldcg(pr + e);
            }
        }
        const int g = r / T, t = r % T;
        IE* dst = og + ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * T + t) * d;
        const float inv = (lim[i] >= 0 && L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) {
            const int e = lane + 32 * c;
            if (e < d) store_out(dst + e, (lim[i] >= 0) ? acc[c] * inv : 0.f);
        }
    }
    if (threadIdx.x == 0) p.counters[unit] = 0;  // ready for the next call
}

template <typename SE, typename IE>
cudaError_t launch_generic(const F32Params& p, cudaStream_t stream) {
    const size_t smem = (static_cast<size_t>(kRows + 2 * kKeys) * p.d + kKeys) * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<SE, IE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(((kRows + 2 * kKeys) * kMaxD + kKeys) * sizeof(float)));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(((p.R + kRows - 1) / kRows) * p.splits, p.Hkv, p.B);
    attn_f32_kernel<SE, IE><<<grid, kWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_f32(const F32Params& p, cudaStream_t stream) {
    if (p.kind == 2) return launch_generic<uint8_t, __nv_bfloat16>(p, stream);
    if (p.kind == 1) return launch_generic<__nv_bfloat16, __nv_bfloat16>(p, stream);
    return launch_generic<float, float>(p, stream);
}

}  // namespace kvc
