// Split-KV GQA attention over the preallocated cache, bf16 storage, d = 128.
//
// What it computes ("Implement grouped-query attention over a preallocated KV
// cache...", "A strong answer", gqa_attention): for every row b, KV head kvh
// and query row r = g*T + t of that head's group (query head kvh*G + g), with
// t < n_new[b], the softmax(q.k / sqrt(d)) weighted sum of V over keys
// 0 .. prior[b] + t, prior = lens - n_new (bottom-right causal offset, "Write
// the causal mask for a decode step...", TL;DR).  Padded queries give 0.
//
// How (GB300):
//  * One persistent CTA per SM.  All (unit, 64-key tile) pairs of the call are
//    numbered and cut into equal contiguous ranges, one per CTA, so ragged row
//    lengths never leave SMs idle; a unit whose tiles straddle CTAs is merged
//    by the last CTA to finish it (per-unit counter, log-sum-exp merge), so
//    the whole call is one launch.
//  * Warp 4 is the producer: one lane streams K and V tiles (64 keys x 128)
//    through TMA (cp.async.bulk.tensor, 128-byte swizzle) into a 4-stage ring
//    guarded by mbarriers.  Each tile is loaded once and serves all G*T query
//    rows of the group (no KV repeat).
//  * Warps 0-3 consume.  With G*T <= 16 rows (decode) the four warps split the
//    tile's keys and merge their softmax states at the end of a unit; with up
//    to 32 or 64 rows they split rows as well.  QK^T and PV run on mma.sync
//    bf16 tiles (16 rows x 8 keys / 8 dims) with fp32 accumulators; softmax is
//    online in base 2 with log2(e)/sqrt(d) folded into one scale.
//  * Tile classification ("Write the causal mask...", tiled-kernel paragraph):
//    a tile whose last key is at or below every valid row's limit is fully
//    visible and skips the mask; tiles past the last visible key are never
//    scheduled; the rest compare key and limit per element.  No mask tensor.
//  * Cache slots past lens may hold anything (stale or NaN).  Masked scores
//    are replaced, never multiplied, and V rows past the unit's last visible
//    key are cleared in shared memory before PV, so 0 * NaN cannot occur.
//  * Every mbarrier wait is bounded in time; on expiry the kernel records an
//    error code in the workspace and finishes instead of hanging.

#include <math.h>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kStages = 4;
constexpr int kD = kHeadDimBf16;
constexpr int kHalfBytes = kKeyTile * 128;   // 64 keys x 64 dims x 2 B (one swizzled box)
constexpr int kTileBytes = 2 * kHalfBytes;   // 64 keys x 128 dims
constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
constexpr int kPartStride = kD + 4;          // floats per partial row: O[128], m, l, pad
constexpr uint64_t kWaitLimitNs = 2000000000ull;

constexpr size_t kObufBytes = 3 * 16 * kD * sizeof(float);
constexpr size_t kMlBytes = kConsumerWarps * 16 * 2 * sizeof(float);
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + kObufBytes + kMlBytes + 2 * kStages * 8 + 16;

__device__ __forceinline__ int cta_of_tile(long long x, long long N, long long P) {
    return static_cast<int>(((x + 1) * P - 1) / N);
}

// Largest q with gstart[q] <= x (gstart nondecreasing, x < gstart[NB]).
__device__ __forceinline__ int locate_group(const DecodeParams& p, int x) {
    int lo = 0, hi = p.NB;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.gstart[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct Cursor {
    int q, kvh, j, nt;
    __device__ __forceinline__ void init(const DecodeParams& p, int x) {
        q = locate_group(p, x);
        nt = (p.gstart[q + 1] - p.gstart[q]) / p.Hkv;
        const int off = x - p.gstart[q];
        kvh = off / nt;
        j = off - kvh * nt;
    }
    __device__ __forceinline__ void advance(const DecodeParams& p) {
        if (++j < nt) return;
        j = 0;
        if (++kvh < p.Hkv) return;
        kvh = 0;
        ++q;
        while (q < p.NB && p.gstart[q + 1] == p.gstart[q]) ++q;
        if (q < p.NB) nt = (p.gstart[q + 1] - p.gstart[q]) / p.Hkv;
    }
};

__device__ __forceinline__ void store_bf16x4(void* dst, float a, float b, float c, float d) {
    uint2 v;
    v.x = ptx::pack_bf16x2(a, b);
    v.y = ptx::pack_bf16x2(c, d);
    *reinterpret_cast<uint2*>(dst) = v;
}

// Merge the partial (m, l, O) of every CTA that worked on unit u and write the
// unit's valid rows of `out`.  Run by the 128 consumer threads of the last CTA.
template <int RPB>
__device__ void merge_unit(const DecodeParams& p, int u, int c0, int c1, int b, int rb, int kvh, int ctid) {
    const int nn = p.n_new[b];
    for (int idx = ctid; idx < RPB * (kD / 4); idx += kConsumerThreads) {
        const int lr = idx >> 5, c4 = idx & 31;
        const int r = rb * RPB + lr;
        if (r >= p.R || (r % p.T) >= nn) continue;
        float mstar = -INFINITY;
        for (int i = c0; i <= c1; ++i) {
            const float* part = p.partials + (static_cast<size_t>(u + i) * RPB + lr) * kPartStride;
            mstar = fmaxf(mstar, __ldcg(part + kD));
        }
        float lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = c0; i <= c1; ++i) {
            const float* part = p.partials + (static_cast<size_t>(u + i) * RPB + lr) * kPartStride;
            const float mi = __ldcg(part + kD);
            const float w = (mi == -INFINITY) ? 0.f : ptx::ex2(mi - mstar);
            lsum += w * __ldcg(part + kD + 1);
            const float4 oi = __ldcg(reinterpret_cast<const float4*>(part) + c4);
            acc.x += w * oi.x;
            acc.y += w * oi.y;
            acc.z += w * oi.z;
            acc.w += w * oi.w;
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const int g = r / p.T, t = r % p.T;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                             ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * p.T + t) * kD + c4 * 4;
        store_bf16x4(dst, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_splitkv_bf16_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                               const __grid_constant__ CUtensorMap tmV) {
    constexpr int KS = kConsumerWarps / MT;  // key slices per tile
    constexpr int KW = kKeyTile / KS;        // keys per warp per tile (16 * MT)
    constexpr int RPB = 16 * MT;             // query rows per block
    constexpr int NBS = KW / 8;              // score n-blocks per warp

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    float* obuf = reinterpret_cast<float*>(smem + kStages * kStageBytes);
    float* ml = obuf + 3 * 16 * kD;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ml + kConsumerWarps * 16 * 2);
    volatile int* flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
    volatile int* abort_flag = flag + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Padded queries (t >= n_new[b]) output zeros; spread over the whole grid.
    {
        const int rows_total = p.B * p.Hq * p.T;
        for (int row = blockIdx.x * kThreads + tid; row < rows_total; row += gridDim.x * kThreads) {
            const int t = row % p.T;
            const int b = row / (p.Hq * p.T);
            if (t >= p.n_new[b]) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * kD);
#pragma unroll
                for (int i = 0; i < kD * 2 / 16; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }

    const long long N = p.total_tiles, P = gridDim.x;
    const int x0 = static_cast<int>(static_cast<long long>(blockIdx.x) * N / P);
    const int x1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * N / P);
    if (x0 >= x1) return;

    const uint32_t stage0 = ptx::smem_addr(stages);
    const uint32_t bar0 = ptx::smem_addr(bars);  // full[s] = bar0 + 8s, empty[s] = bar0 + 8(kStages + s)
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar0 + 8 * s, 1);
            ptx::mbar_init(bar0 + 8 * (kStages + s), kConsumerWarps);
        }
        *flag = 0;
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();

    // ------------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tmK);
            ptx::tma_prefetch_desc(&tmV);
            Cursor cur;
            cur.init(p, x0);
            int issued = 0;
            for (int x = x0, it = 0; x < x1; ++x, ++it) {
                const int s = it % kStages;
                if (it >= kStages) {
                    if (!ptx::mbar_wait_bounded(bar0 + 8 * (kStages + s), ((it / kStages) & 1) ^ 1, kWaitLimitNs)) {
                        atomicExch(p.err, kDevTimeoutEmpty);
                        *abort_flag = 1;
                    }
                }
                if (*abort_flag) break;  // the producer is in no named barrier, so it may stop early
                const int b = cur.q / p.RB;
                const int row = (b * p.Hkv + cur.kvh) * p.max_len + cur.j * kKeyTile;
                const uint32_t full = bar0 + 8 * s;
                const uint32_t sK = stage0 + s * kStageBytes;
                ptx::mbar_arrive_expect_tx(full, kStageBytes);
                ptx::tma_load_2d(sK, &tmK, 0, row, full);
                ptx::tma_load_2d(sK + kHalfBytes, &tmK, 64, row, full);
                ptx::tma_load_2d(sK + kTileBytes, &tmV, 0, row, full);
                ptx::tma_load_2d(sK + kTileBytes + kHalfBytes, &tmV, 64, row, full);
                ++issued;
                cur.advance(p);
            }
            // Never leave the CTA with copies in flight: wait (bounded) for the
            // last phase armed on every stage.  In a clean run these phases
            // have already completed and the waits return at once.
            for (int it = max(0, issued - kStages); it < issued; ++it) {
                if (!ptx::mbar_wait_bounded(bar0 + 8 * (it % kStages), (it / kStages) & 1, kWaitLimitNs)) {
                    atomicExch(p.err, kDevTimeoutDrain);
                    break;
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int mt = warp % MT, ks = warp / MT;
    const int quad = lane & 3;
    const int lrow0 = mt * 16 + (lane >> 2);  // this thread's block rows: lrow0, lrow0 + 8

    Cursor cur;
    cur.init(p, x0);

    float o[16][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    uint32_t qa[8][4];
    int lim0 = -1, lim1 = -1, min_lim = 0, extent = 0, seg_j0 = 0;

    for (int x = x0, it = 0; x < x1; ++x, ++it) {
        const int s = it % kStages;
        const int b = cur.q / p.RB, rb = cur.q - (cur.q / p.RB) * p.RB;
        const int j = cur.j, nt = cur.nt, kvh = cur.kvh;

        if (x == x0 || j == 0) {
            // New unit segment: row limits, extent, query fragments, fresh state.
            const int prior = p.prior[b], nn = p.n_new[b];
            min_lim = 0x7fffffff;
            extent = 0;
            for (int i = 0; i < RPB; ++i) {
                const int r = rb * RPB + i;
                if (r >= p.R) break;
                const int t = r % p.T;
                if (t < nn) {
                    min_lim = min(min_lim, prior + t);
                    extent = max(extent, prior + t + 1);
                }
            }
            seg_j0 = j;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = rb * RPB + lrow0 + 8 * h;
                int lim = -1;
                const __nv_bfloat16* qrow = nullptr;
                if (r < p.R) {
                    const int g = r / p.T, t = r % p.T;
                    if (t < nn) lim = prior + t;
                    qrow = static_cast<const __nv_bfloat16*>(p.q) +
                           ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * p.T + t) * kD;
                }
                if (h == 0) lim0 = lim; else lim1 = lim;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    qa[kk][h] = qrow ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * quad) : 0u;
                    qa[kk][2 + h] = qrow ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * quad) : 0u;
                }
            }
#pragma unroll
            for (int nb = 0; nb < 16; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }

        // On expiry the warp records the error and carries on with whatever the
        // stage holds (the call's output is then invalid): consumer warps meet
        // at named barriers, so none may leave the loop alone.  After the first
        // expiry further waits try once only.
        if (!ptx::mbar_wait_bounded(bar0 + 8 * s, (it / kStages) & 1, *abort_flag ? 0ull : kWaitLimitNs)) {
            atomicExch(p.err, kDevTimeoutFull);
            *abort_flag = 1;
        }

        const uint32_t sK = stage0 + s * kStageBytes;
        const uint32_t sV = sK + kTileBytes;
        const int tile0 = j * kKeyTile;

        if (tile0 + kKeyTile > extent) {
            // Clear V rows at or past the unit's last visible key (slots past
            // lens may hold NaN; their probabilities are 0 but 0 * NaN is NaN).
            const int vr0 = extent - tile0;
            const int per_half = (kKeyTile - vr0) * 8;
            uint8_t* vbase = stages + s * kStageBytes + kTileBytes;
            for (int idx = tid; idx < 2 * per_half; idx += kConsumerThreads) {
                const int hf = idx / per_half, rem = idx - hf * per_half;
                *reinterpret_cast<uint4*>(vbase + hf * kHalfBytes + (vr0 + (rem >> 3)) * 128 + (rem & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            ptx::fence_proxy_async_smem();
            ptx::named_barrier_sync(1, kConsumerThreads);
        }
        const bool full_tile = (tile0 + kKeyTile - 1 <= min_lim);

        // S = Q K^T for this warp's 16 rows x KW keys.
        float sc[NBS][4];
#pragma unroll
        for (int nb = 0; nb < NBS; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int kb = 0; kb < MT; ++kb) {
                const int mi = lane >> 3;
                const int key = ks * KW + kb * 16 + (mi >> 1) * 8 + (lane & 7);
                const int chunk = 2 * kk + (mi & 1);
                const uint32_t addr = sK + (chunk >> 3) * kHalfBytes + key * 128 + (((chunk & 7) ^ (key & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ptx::ldmatrix_x4(addr, b0, b1, b2, b3);
                ptx::mma_bf16_16816(sc[2 * kb], qa[kk], b0, b1);
                ptx::mma_bf16_16816(sc[2 * kb + 1], qa[kk], b2, b3);
            }
        }

        // Mask (diagonal / ragged tiles only) and online softmax in base 2.
        const int kbase = tile0 + ks * KW + 2 * quad;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nb = 0; nb < NBS; ++nb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = sc[nb][e] * p.scale_log2;
                if (!full_tile) {
                    const int key = kbase + nb * 8 + (e & 1);
                    if (key > ((e < 2) ? lim0 : lim1)) v = -INFINITY;
                }
                sc[nb][e] = v;
            }
            mx0 = fmaxf(mx0, fmaxf(sc[nb][0], sc[nb][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[nb][2], sc[nb][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float al0 = ptx::ex2(m0 - mu0), al1 = ptx::ex2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nb = 0; nb < NBS; ++nb) {
            sc[nb][0] = ptx::ex2(sc[nb][0] - mu0);
            sc[nb][1] = ptx::ex2(sc[nb][1] - mu0);
            sc[nb][2] = ptx::ex2(sc[nb][2] - mu1);
            sc[nb][3] = ptx::ex2(sc[nb][3] - mu1);
            ps0 += sc[nb][0] + sc[nb][1];
            ps1 += sc[nb][2] + sc[nb][3];
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int nb = 0; nb < 16; ++nb) {
            o[nb][0] *= al0;
            o[nb][1] *= al0;
            o[nb][2] *= al1;
            o[nb][3] *= al1;
        }

        // O += P V.
#pragma unroll
        for (int kb = 0; kb < MT; ++kb) {
            uint32_t a[4];
            a[0] = ptx::pack_bf16x2(sc[2 * kb][0], sc[2 * kb][1]);
            a[1] = ptx::pack_bf16x2(sc[2 * kb][2], sc[2 * kb][3]);
            a[2] = ptx::pack_bf16x2(sc[2 * kb + 1][0], sc[2 * kb + 1][1]);
            a[3] = ptx::pack_bf16x2(sc[2 * kb + 1][2], sc[2 * kb + 1][3]);
#pragma unroll
            for (int dc = 0; dc < 8; ++dc) {
                const int mi = lane >> 3;
                const int key = ks * KW + kb * 16 + (mi & 1) * 8 + (lane & 7);
                const int chunk = 2 * dc + (mi >> 1);
                const uint32_t addr = sV + (chunk >> 3) * kHalfBytes + key * 128 + (((chunk & 7) ^ (key & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ptx::ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                ptx::mma_bf16_16816(o[2 * dc], a, b0, b1);
                ptx::mma_bf16_16816(o[2 * dc + 1], a, b2, b3);
            }
        }

        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar0 + 8 * (kStages + s));

        const bool seg_end = (x == x1 - 1) || (j == nt - 1);
        if (seg_end) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            if (KS > 1) {
                // Merge the key slices' softmax states into the ks == 0 warps.
                const int r0 = lane >> 2;
                if (quad == 0) {
                    ml[(warp * 16 + r0) * 2 + 0] = m0;
                    ml[(warp * 16 + r0) * 2 + 1] = l0;
                    ml[(warp * 16 + r0 + 8) * 2 + 0] = m1;
                    ml[(warp * 16 + r0 + 8) * 2 + 1] = l1;
                }
                ptx::named_barrier_sync(1, kConsumerThreads);
                float mf0 = -INFINITY, mf1 = -INFINITY;
#pragma unroll
                for (int k2 = 0; k2 < KS; ++k2) {
                    const int w2 = mt + k2 * MT;
                    mf0 = fmaxf(mf0, ml[(w2 * 16 + r0) * 2]);
                    mf1 = fmaxf(mf1, ml[(w2 * 16 + r0 + 8) * 2]);
                }
                const float mfu0 = (mf0 == -INFINITY) ? 0.f : mf0;
                const float mfu1 = (mf1 == -INFINITY) ? 0.f : mf1;
                float lf0 = 0.f, lf1 = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < KS; ++k2) {
                    const int w2 = mt + k2 * MT;
                    lf0 += ml[(w2 * 16 + r0) * 2 + 1] * ptx::ex2(ml[(w2 * 16 + r0) * 2] - mfu0);
                    lf1 += ml[(w2 * 16 + r0 + 8) * 2 + 1] * ptx::ex2(ml[(w2 * 16 + r0 + 8) * 2] - mfu1);
                }
                const float f0 = ptx::ex2(m0 - mfu0), f1 = ptx::ex2(m1 - mfu1);
#pragma unroll
                for (int nb = 0; nb < 16; ++nb) {
                    o[nb][0] *= f0;
                    o[nb][1] *= f0;
                    o[nb][2] *= f1;
                    o[nb][3] *= f1;
                }
                if (ks > 0) {
                    float* ob = obuf + ((ks - 1) * MT + mt) * 16 * kD;
#pragma unroll
                    for (int nb = 0; nb < 16; ++nb) {
                        const int col = nb * 8 + 2 * quad;
                        *reinterpret_cast<float2*>(ob + r0 * kD + col) = make_float2(o[nb][0], o[nb][1]);
                        *reinterpret_cast<float2*>(ob + (r0 + 8) * kD + col) = make_float2(o[nb][2], o[nb][3]);
                    }
                }
                ptx::named_barrier_sync(1, kConsumerThreads);
                if (ks == 0) {
#pragma unroll
                    for (int k2 = 1; k2 < KS; ++k2) {
                        const float* ob = obuf + ((k2 - 1) * MT + mt) * 16 * kD;
#pragma unroll
                        for (int nb = 0; nb < 16; ++nb) {
                            const int col = nb * 8 + 2 * quad;
                            const float2 a = *reinterpret_cast<const float2*>(ob + r0 * kD + col);
                            const float2 c = *reinterpret_cast<const float2*>(ob + (r0 + 8) * kD + col);
                            o[nb][0] += a.x;
                            o[nb][1] += a.y;
                            o[nb][2] += c.x;
                            o[nb][3] += c.y;
                        }
                    }
                }
                m0 = mf0;
                m1 = mf1;
                l0 = lf0;
                l1 = lf1;
                ptx::named_barrier_sync(1, kConsumerThreads);
            }

            const int u = cur.q * p.Hkv + kvh;
            const bool sole = (seg_j0 == 0) && (j == nt - 1);
            if (sole) {
                if (ks == 0) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int lim = h ? lim1 : lim0;
                        if (lim < 0) continue;
                        const int r = rb * RPB + lrow0 + 8 * h;
                        const int g = r / p.T, t = r % p.T;
                        const float l = h ? l1 : l0;
                        const float inv = l > 0.f ? 1.f / l : 0.f;
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                                             ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * p.T + t) * kD;
#pragma unroll
                        for (int nb = 0; nb < 16; ++nb) {
                            const int col = nb * 8 + 2 * quad;
                            *reinterpret_cast<uint32_t*>(dst + col) =
                                ptx::pack_bf16x2(o[nb][2 * h] * inv, o[nb][2 * h + 1] * inv);
                        }
                    }
                }
            } else {
                const int slot = u + blockIdx.x;
                if (ks == 0) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float* part = p.partials + (static_cast<size_t>(slot) * RPB + lrow0 + 8 * h) * kPartStride;
#pragma unroll
                        for (int nb = 0; nb < 16; ++nb) {
                            const int col = nb * 8 + 2 * quad;
                            __stcg(reinterpret_cast<float2*>(part + col), make_float2(o[nb][2 * h], o[nb][2 * h + 1]));
                        }
                        if (quad == 0) {
                            __stcg(part + kD, h ? m1 : m0);
                            __stcg(part + kD + 1, h ? l1 : l0);
                        }
                    }
                }
                __threadfence();
                ptx::named_barrier_sync(1, kConsumerThreads);
                if (tid == 0) {
                    const long long us = static_cast<long long>(p.gstart[cur.q]) + static_cast<long long>(kvh) * nt;
                    const int c0 = cta_of_tile(us, N, P), c1 = cta_of_tile(us + nt - 1, N, P);
                    const int old = atomicAdd(p.counters + u, 1);
                    if (old == c1 - c0) {
                        p.counters[u] = 0;  // all contributors arrived: leave it clean for the next call
                        *flag = c0 + 1;
                    } else {
                        *flag = 0;
                    }
                }
                ptx::named_barrier_sync(1, kConsumerThreads);
                const int f = *flag;
                if (f) {
                    __threadfence();
                    const long long us = static_cast<long long>(p.gstart[cur.q]) + static_cast<long long>(kvh) * nt;
                    const int c1 = cta_of_tile(us + nt - 1, N, P);
                    merge_unit<RPB>(p, u, f - 1, c1, b, rb, kvh, tid);
                }
                ptx::named_barrier_sync(1, kConsumerThreads);
            }
        }
        cur.advance(p);
    }
}

template <int MT>
cudaError_t launch_mt(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int grid,
                      cudaStream_t stream) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_splitkv_bf16_kernel<MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    decode_splitkv_bf16_kernel<MT><<<grid, kThreads, kSmemBytes, stream>>>(p, tmK, tmV);
    return cudaGetLastError();
}

__global__ void wait_selftest_kernel(int* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on this barrier: the wait must give up by itself.
        if (!ptx::mbar_wait_bounded(ptx::smem_addr(&bar), 0, limit_ns)) atomicExch(err, kDevTimeoutTest);
    }
}

}  // namespace

DecodeLaunch decode_launch_shape(int mt) { return DecodeLaunch{mt, kThreads, kSmemBytes}; }

cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int mt,
                               int grid, cudaStream_t stream) {
    switch (mt) {
        case 1: return launch_mt<1>(p, tmK, tmV, grid, stream);
        case 2: return launch_mt<2>(p, tmK, tmV, grid, stream);
        case 4: return launch_mt<4>(p, tmK, tmV, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace kvc
