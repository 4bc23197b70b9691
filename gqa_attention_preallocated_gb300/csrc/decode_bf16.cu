// Split-KV GQA attention over the preallocated cache, bf16 or FP8 E4M3
// storage, d = 128.
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
//    lengths never leave SMs idle.  A unit finished by one writer is written
//    straight to `out`; otherwise every writer (a CTA, or with warps owning
//    whole tiles every warp that took some of its tiles) leaves a partial
//    (m, l, O), merged by the small combine kernel that follows in the stream
//    (log-sum-exp merge).  Launches are chained with programmatic dependent
//    launch, so a kernel's launch and prologue overlap the previous kernel's
//    tail.
//  * Warp 4 is the producer: one lane streams K and V tiles (64 keys x 128)
//    through TMA (cp.async.bulk.tensor, 128-byte swizzle) into a ring of
//    stages guarded by mbarriers.  Each tile is loaded once and serves all G*T
//    query rows of the group (no KV repeat).
//  * Warps 0-3 consume.  With G*T <= 16 rows (decode, short verify) each warp
//    owns whole tiles in turn (tile i goes to warp i mod 4) and keeps its own
//    softmax state, so four tiles are in flight at once and each warp runs
//    eight independent MMA chains per tile; the warps' states merge in the
//    combine kernel.  With up to 32 or 64 rows the warps split rows (and
//    keys).
//    QK^T and PV run on mma.sync bf16 tiles (16 rows x 8 keys / 8 dims) with
//    fp32 accumulators; softmax is online in base 2 with log2(e)/sqrt(d)
//    folded into one scale.
//  * Tile classification ("Write the causal mask...", tiled-kernel paragraph):
//    a tile whose last key is at or below every valid row's limit is fully
//    visible and skips the mask; tiles past the last visible key are never
//    scheduled; the rest compare key and limit per element.  No mask tensor.
//  * Cache slots past lens may hold anything (stale or NaN).  Masked scores
//    are replaced, never multiplied, and V rows past the unit's last visible
//    key are cleared in shared memory before PV, so 0 * NaN cannot occur.
//  * FP8 E4M3 storage ("16. Prefill, decode and the KV cache", exercise 4;
//    template argument F8): 64-key tiles of one byte a value, converted to f16
//    exactly in registers (one cvt per pair) and multiplied by f16 queries,
//    with the head dimension permuted so each thread's K bytes are contiguous
//    and the output columns permuted so its V bytes are one 16-byte chunk per
//    key; the per-head K scale folds into the softmax scale, the V scale into
//    the output.  Appends fused into the launch quantize the new rows.
//  * Every wait is bounded in time; on expiry the kernel records an error code
//    in the workspace and finishes instead of hanging.

#include <math.h>

#include <utility>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kConsumerWarps = 4;  // consumer warps, except FP8 caches with warps owning whole tiles
// Head dimensions: D = 128 (bf16 and FP8 storage) and D = 64 (bf16).  A TMA
// box is 64 keys x 128 bytes (64 bf16 columns, or 128 E4M3 codes) with the
// 128-byte swizzle; a bf16 tile of 64 keys is D / 64 boxes.
// floats per partial row: O[D], m, l, pad
__host__ __device__ constexpr int part_stride(int D) { return D + 4; }
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLazyRescale = 8.0f;  // log2 of the largest factor p may reach above the reference
constexpr size_t kMlBytes = kConsumerWarps * 16 * 2 * sizeof(float);

// Compile-time shape of the kernel for MT m-tiles (16 query rows each).
//
// Warps that own whole tiles (MT = 1) never meet: each writes its own partial
// softmax state of a unit to the workspace and the combine kernel merges them,
// so no shared merge buffer is needed and the ring gets a seventh stage.  With
// MT = 2 or 4 the warps split every tile and merge their states in shared
// memory at the end of a unit.
template <int MT, bool F8, int D>
struct Shape {
    static_assert(D == 128 || (D == 64 && !F8), "head dimensions: 128 (bf16, FP8) and 64 (bf16)");
    static constexpr bool kTilePar = (MT == 1);                // warps own whole tiles
    // Keys per tile: 64, or 128 for 64-wide heads, whose 64-key tile would
    // carry half the bytes of a 128-wide one for the same per-tile work.
    static constexpr int kKeyTile = key_tile_keys(D, F8);
    static constexpr int kHalfBytes = kKeyTile * 128;  // one swizzled box: kKeyTile rows x 128 bytes
    // bytes of one K (or V) tile: D / 64 boxes of bf16, or one 128-byte-row
    // box of E4M3 codes
    static constexpr int kTileB = F8 ? kKeyTile * 128 : kKeyTile * D * 2;
    static constexpr int kStageB = 2 * kTileB;
    // as many stages as fit: 224 KB (7 of 32 KB, 14 of 16 KB) with warps owning
    // tiles, 128 KB beside the shared merge buffers otherwise
    static constexpr int kStages = (kTilePar ? 229376 : 131072) / kStageB;
    // Consumer warps: with FP8 storage (or 64-wide heads) a tile holds half the
    // bytes for the same per-tile work, so one warp per SM sub-partition cannot
    // keep up with HBM; seven tile-owning warps (two per sub-partition, with
    // the producer) hide each other's latency.
    static constexpr int kCW = ((F8 || D == 64) && kTilePar) ? 7 : kConsumerWarps;
    static constexpr int kCT = kCW * 32;
    static constexpr int kThreads = kCT + 32;
    static constexpr int kKeySlices = kTilePar ? 1 : kCW / MT;
    static constexpr int kKW = kKeyTile / kKeySlices;          // keys per warp per tile
    // Keys per pass over the tile: an FP8 warp's registers hold the scores of
    // 64 keys, so it takes a 128-key tile in two passes.
    static constexpr int kKWP = (F8 && kKW > 64) ? 64 : kKW;
    static constexpr int kMerge = kTilePar ? 1 : kKeySlices;   // states per m-tile merged in shared memory
    static constexpr int kWays = kTilePar ? kCW : 1;  // partial sub-slots per (unit, CTA)
    static constexpr int kRPB = 16 * MT;
    static constexpr int kEmptyCount = kTilePar ? 1 : kCW;
    static constexpr size_t kObuf = kTilePar ? 0 : 3 * 16 * D * sizeof(float);
    static constexpr size_t kMl = kTilePar ? 0 : kMlBytes;
    static constexpr size_t kSmem = 1024 + kStages * kStageB + kObuf + kMl + 2 * kStages * 8 + (kStages + 4) * 4;
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

// The call's work partition, read only after the grid-dependency wait.
// Part<false>: planned on the host, in the kernel parameters (indexed in
// parameter space).  Part<true>: planned on the device from device-resident
// lengths (a DevicePlan in the workspace).
template <bool DP>
struct Part;

template <>
struct Part<false> {
    const DecodeParams& p;
    __device__ __forceinline__ int gstart(int i) const { return p.gstart[i]; }
    __device__ __forceinline__ int prior(int b) const { return p.prior[b]; }
    __device__ __forceinline__ int n_new(int b) const { return p.n_new[b]; }
    __device__ __forceinline__ int total_tiles() const { return p.total_tiles; }
    __device__ __forceinline__ int NB() const { return p.NB; }
    __device__ __forceinline__ int Hkv() const { return p.Hkv; }
};

template <>
struct Part<true> {
    const DecodeParams& p;
    __device__ __forceinline__ int gstart(int i) const { return p.dplan->gstart[i]; }
    __device__ __forceinline__ int prior(int b) const { return p.dplan->prior[b]; }
    __device__ __forceinline__ int n_new(int b) const { return p.dplan->n_new[b]; }
    __device__ __forceinline__ int total_tiles() const { return p.dplan->total_tiles; }
    __device__ __forceinline__ int NB() const { return p.NB; }
    __device__ __forceinline__ int Hkv() const { return p.Hkv; }
};

// First key tile (absolute position / 64) of group q's units: 0, or with a
// window the tile holding the window start of the block's earliest query
// (the same rule as the planners'; tiles before it are never scheduled).
template <bool DP, int KT>
__device__ __forceinline__ int first_tile(const Part<DP>& w, int q) {
    const DecodeParams& p = w.p;
    if (p.window <= 0) return 0;
    const int b = q / p.RB, rb = q - b * p.RB;
    const int prior = w.prior(b), nn = w.n_new(b);
    const int r0 = rb * p.RPB, r1 = min(p.R, r0 + p.RPB);
    int qmin = 0x7fffffff;
    if (r1 - r0 >= p.T) {
        if (nn > 0) qmin = prior;
    } else {
        for (int r = r0; r < r1; ++r)
            if (r % p.T < nn) qmin = min(qmin, prior + r % p.T);
    }
    return qmin == 0x7fffffff ? 0 : max(0, qmin - p.window + 1) / KT;
}

// Largest q with gstart[q] <= x (gstart nondecreasing, x < gstart[NB]).
template <bool DP>
__device__ __forceinline__ int locate_group(const Part<DP>& w, int x) {
    int lo = 0, hi = w.NB();
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (w.gstart(mid) <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <bool DP, int KT>
struct Cursor {
    int q, kvh, j, nt, t0;  // t0: the group's first key tile
    __device__ __forceinline__ void init(const Part<DP>& w, int x) {
        q = locate_group(w, x);
        nt = (w.gstart(q + 1) - w.gstart(q)) / w.Hkv();
        const int off = x - w.gstart(q);
        kvh = off / nt;
        j = off - kvh * nt;
        t0 = first_tile<DP, KT>(w, q);
    }
    __device__ __forceinline__ void advance(const Part<DP>& w) {
        if (++j < nt) return;
        j = 0;
        if (++kvh < w.Hkv()) return;
        kvh = 0;
        ++q;
        while (q < w.NB() && w.gstart(q + 1) == w.gstart(q)) ++q;
        if (q < w.NB()) {
            nt = (w.gstart(q + 1) - w.gstart(q)) / w.Hkv();
            t0 = first_tile<DP, KT>(w, q);
        }
    }
};

// Row (of the cache's 2-D view) of the key at absolute position a of unit
// (b, kvh): contiguous, ring (a mod max_len) or paged (through the block
// table).  Tiles never straddle a ring wrap or a page (max_len / page are
// multiples of the tile size there).  A bad table entry records an error.
__device__ __forceinline__ int key_row(const DecodeParams& p, int b, int kvh, int a) {
    bool bad = false;
    const int row = phys_row(p.pg, p.ring, p.Hkv, p.max_len, b, kvh, a, &bad);
    if (bad) atomicExch(p.err, kDevBadPage);
    return row;
}

// bf16 pair -> f16 pair (exact for |x| in f16's range: bf16 has fewer
// significant bits); used for the queries of an FP8 cache's f16 MMAs.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return ptx::pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ void store_bf16x4(void* dst, float a, float b, float c, float d) {
    uint2 v;
    v.x = ptx::pack_bf16x2(a, b);
    v.y = ptx::pack_bf16x2(c, d);
    *reinterpret_cast<uint2*>(dst) = v;
}

// Wait until the producer has claimed stage s for tile `it` (bounded).
__device__ __forceinline__ bool wait_stage_tag(const volatile int* tag, int it, uint64_t limit_ns) {
    if (*tag == it) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (*tag == it) return true;
        if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// MT: m-tiles of 16 query rows; DP: the partition comes from a device plan;
// TREE: draft-tree ancestor masks apply (compiled out otherwise).
template <int MT, bool DP, bool TREE, bool F8, int D>
__global__ void __launch_bounds__(Shape<MT, F8, D>::kThreads, 1)
    decode_splitkv_bf16_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                               const __grid_constant__ CUtensorMap tmV) {
    using S = Shape<MT, F8, D>;
    constexpr int KT = S::kKeyTile;  // keys per tile
    constexpr int PS = part_stride(D);
    constexpr int CPR = D / 8;  // 16-byte chunks of a bf16 row
    constexpr int kStages = S::kStages;
    constexpr int KW = S::kKW;
    constexpr int RPB = S::kRPB;
    constexpr int KWP = S::kKWP;  // keys per pass (KW / KWP passes per tile)
    constexpr int NBS = KWP / 8;  // score n-blocks per warp per pass
    constexpr int KB = KWP / 16;  // 16-key blocks per warp per pass
    constexpr int NM = S::kMerge;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    float* obuf = reinterpret_cast<float*>(smem + kStages * S::kStageB);
    float* ml = reinterpret_cast<float*>(smem + kStages * S::kStageB + S::kObuf);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * S::kStageB + S::kObuf + S::kMl);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
    volatile int* stage_tag = abort_flag + 4;  // tile index the producer last put in each stage

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Part<DP> wp{p};
    // This CTA's tiles (host plan: known before the dependency wait).
    long long N = DP ? 0 : wp.total_tiles();
    const long long P = gridDim.x;
    int x0 = static_cast<int>(static_cast<long long>(blockIdx.x) * N / P);
    int x1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * N / P);

    // Prologue: touches no memory that earlier work in the stream may write.
    const uint32_t stage0 = ptx::smem_addr(stages);
    const uint32_t bar0 = ptx::smem_addr(bars);  // full[s] = bar0 + 8s, empty[s] = bar0 + 8(kStages + s)
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar0 + 8 * s, 1);
            ptx::mbar_init(bar0 + 8 * (kStages + s), S::kEmptyCount);
            stage_tag[s] = -1;
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == S::kCW && lane == 0) {
        ptx::tma_prefetch_desc(&tmK);
        ptx::tma_prefetch_desc(&tmV);
    }
    __syncthreads();
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    if (DP) {
        if (p.dplan->skip) return;  // a rejected device-resident step: nothing is written
        N = wp.total_tiles();
        x0 = static_cast<int>(static_cast<long long>(blockIdx.x) * N / P);
        x1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * N / P);
    }

    // Padded queries (t >= n_new[b]) output zeros; spread over the whole grid.
    {
        const int rows_total = p.B * p.Hq * p.T;
        for (int row = blockIdx.x * S::kThreads + tid; row < rows_total; row += gridDim.x * S::kThreads) {
            const int t = row % p.T;
            const int b = row / (p.Hq * p.T);
            if (t >= wp.n_new(b)) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * D);
#pragma unroll
                for (int i = 0; i < CPR; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    if (x0 >= x1) return;

    // ------------------------------------------------------------------ producer
    if (warp == S::kCW) {
        if (lane == 0) {
            Cursor<DP, KT> cur;
            cur.init(wp, x0);
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
                const int row = key_row(p, b, cur.kvh, (cur.t0 + cur.j) * KT);
                const uint32_t full = bar0 + 8 * s;
                const uint32_t sK = stage0 + s * S::kStageB;
                stage_tag[s] = it;
                ptx::mbar_arrive_expect_tx(full, S::kStageB);
                if constexpr (F8) {  // one 64-row x 128-byte box each
                    ptx::tma_load_2d(sK, &tmK, 0, row, full);
                    ptx::tma_load_2d(sK + S::kTileB, &tmV, 0, row, full);
                } else {
#pragma unroll
                    for (int hf = 0; hf < D / 64; ++hf) {  // 64-column boxes of the K and V tiles
                        ptx::tma_load_2d(sK + hf * S::kHalfBytes, &tmK, 64 * hf, row, full);
                        ptx::tma_load_2d(sK + S::kTileB + hf * S::kHalfBytes, &tmV, 64 * hf, row, full);
                    }
                }
                ++issued;
                cur.advance(wp);
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
    // mt: this warp's m-tile; ms: its index among the NM softmax states of that
    // m-tile merged at a unit's end; koff: first key of its slice of a tile.
    const int mt = S::kTilePar ? 0 : warp % MT;
    const int ms = S::kTilePar ? warp : warp / MT;
    const int koff = S::kTilePar ? 0 : ms * KW;
    const int quad = lane & 3;
    const int lrow0 = mt * 16 + (lane >> 2);  // this thread's block rows: lrow0, lrow0 + 8

    Cursor<DP, KT> cur;
    cur.init(wp, x0);

    float o[D / 8][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    uint32_t qa[D / 16][4];
    int lim0 = -1, lim1 = -1, min_lim = 0, extent = 0, seg_j0 = 0, seg_tiles = 0;
    // Window lower bounds (keys <= lo are outside the window): this thread's
    // two rows, and the largest and smallest over the block's valid rows.
    int lo0 = -1, lo1 = -1, max_lo = -1, min_lo = -1;
    int seg_prior = 0, seg_nn = 0;
    float sl2 = p.scale_log2;  // score scale in base 2 (times the K scale of an FP8 cache)
    // first appended row, lane's 16-byte chunk (K: lanes 0 .. CPR-1, V: CPR .. 2*CPR-1)
    uint4 new_row0 = make_uint4(0u, 0u, 0u, 0u);

    for (int x = x0, it = 0; x < x1; ++x, ++it) {
        const int s = it % kStages;
        const int b = cur.q / p.RB, rb = cur.q - (cur.q / p.RB) * p.RB;
        const int j = cur.j, nt = cur.nt, kvh = cur.kvh;

        if (x == x0 || j == 0) {
            // New unit segment: row limits, extent, query fragments, fresh state.
            const int prior = wp.prior(b), nn = wp.n_new(b);
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
            // With a window the block's rows see keys lim - W < a <= lim.
            max_lo = (p.window > 0 && extent > 0) ? extent - 1 - p.window : -1;
            min_lo = (p.window > 0 && extent > 0) ? min_lim - p.window : -1;
            seg_j0 = j;
            seg_tiles = 0;
            seg_prior = prior;
            seg_nn = nn;
            if constexpr (F8) sl2 = p.scale_log2 * p.kscale[kvh];
            if (S::kTilePar && p.append_new && nn > 0 && lane < 2 * CPR) {
                const uint8_t* src = static_cast<const uint8_t*>((lane < CPR) ? p.k_new : p.v_new) +
                                     (static_cast<size_t>(b) * p.Hkv + kvh) * p.Tn * (D * 2) + (lane % CPR) * 16;
                new_row0 = __ldg(reinterpret_cast<const uint4*>(src));
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = rb * RPB + lrow0 + 8 * h;
                int lim = -1;
                const __nv_bfloat16* qrow = nullptr;
                if (r < p.R) {
                    const int g = r / p.T, t = r % p.T;
                    if (t < nn) lim = prior + t;
                    qrow = static_cast<const __nv_bfloat16*>(p.q) +
                           ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * p.T + t) * D;
                }
                if (h == 0) lim0 = lim; else lim1 = lim;
                const int lo = (p.window > 0 && lim >= 0) ? lim - p.window : -1;
                if (h == 0) lo0 = lo; else lo1 = lo;
                if constexpr (F8) {
                    // f16 fragments with the head dimension permuted: MMA
                    // k-step kk's logical columns 2*quad + {0, 1} and
                    // 2*quad + {8, 9} read d = 32*quad + 4*kk + {0, 1} and
                    // + {2, 3}, so each thread's K bytes are 32 consecutive ones.
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 w = qrow ? __ldg(reinterpret_cast<const uint4*>(qrow + 32 * quad) + c)
                                             : make_uint4(0u, 0u, 0u, 0u);
                        qa[2 * c][h] = bf16x2_to_f16x2(w.x);
                        qa[2 * c][2 + h] = bf16x2_to_f16x2(w.y);
                        qa[2 * c + 1][h] = bf16x2_to_f16x2(w.z);
                        qa[2 * c + 1][2 + h] = bf16x2_to_f16x2(w.w);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        qa[kk][h] = qrow ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * quad) : 0u;
                        qa[kk][2 + h] = qrow ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * quad) : 0u;
                    }
                }
            }
#pragma unroll
            for (int nb = 0; nb < D / 8; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }

        const bool mine = S::kTilePar ? ((it % S::kCW) == warp) : true;
        if (mine) {
            ++seg_tiles;
            // On expiry the warp records the error and carries on with whatever
            // the stage holds (the call's output is then invalid): consumer warps
            // meet at named barriers, so none may leave the loop alone.  After
            // the first expiry further waits try once only.
            const uint64_t limit = *abort_flag ? 0ull : kWaitLimitNs;
            if (S::kTilePar) {
                // With warps taking tiles in turn, the warp that owns tile `it`
                // may reach stage s while an earlier tile of another warp still
                // occupies it.  The mbarrier parity cannot tell phases two apart,
                // so first wait until the producer has put tile `it` in stage s.
                if (!wait_stage_tag(stage_tag + s, it, limit)) {
                    atomicExch(p.err, kDevTimeoutTag);
                    *abort_flag = 1;
                }
            }
            if (!ptx::mbar_wait_bounded(bar0 + 8 * s, (it / kStages) & 1, limit)) {
                atomicExch(p.err, kDevTimeoutFull);
                *abort_flag = 1;
            }

            const uint32_t sK = stage0 + s * S::kStageB;
            const uint32_t sV = sK + S::kTileB;
            const int tile0 = (cur.t0 + j) * KT;  // first key position of the tile

            if (S::kTilePar && p.append_new) {
                // In-kernel append: rows prior .. prior+n_new-1 of this unit that
                // fall in this tile come from k_new / v_new.  The staged copy of
                // those cache slots is stale, so patch it, and write the rows to
                // the cache (this tile is processed exactly once).
                const int lo = max(seg_prior, tile0), hi = min(seg_prior + seg_nn, tile0 + KT);
                if (lo < hi) {
                    // lanes 0 .. CPR-1 write K, CPR .. 2*CPR-1 V, one 16-byte chunk of
                    // the bf16 source row each (the rest idle: D = 64)
                    const int chunk = lane % CPR;
                    const bool is_v = lane >= CPR;
                    const int hi_l = (lane < 2 * CPR) ? hi : lo;
                    const size_t unit = static_cast<size_t>(b) * p.Hkv + kvh;
                    const uint8_t* src = static_cast<const uint8_t*>(is_v ? p.v_new : p.k_new) + unit * p.Tn * (D * 2);
                    uint8_t* dst = static_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache);
                    bool bad = false;
                    const int row0 = phys_row(p.pg, p.ring, p.Hkv, p.max_len, b, kvh, tile0, &bad) - tile0;  // the tile's rows are contiguous
                    if constexpr (F8) {
                        // quantize: code of x * (1/scale), 8 values -> 8 bytes at
                        // bytes 8*chunk .. of the 128-byte row
                        const float inv = __frcp_rn(is_v ? p.vscale[kvh] : p.kscale[kvh]);
                        uint8_t* stg = stages + s * S::kStageB + (is_v ? S::kTileB : 0);
                        for (int pos = lo; pos < hi_l; ++pos) {
                            const int t = pos - seg_prior, r = pos - tile0;
                            const uint4 val = (t == 0) ? new_row0
                                                       : __ldg(reinterpret_cast<const uint4*>(src + t * (D * 2) + chunk * 16));
                            const uint32_t w[4] = {val.x, val.y, val.z, val.w};
                            uint32_t c[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                c[i] = ptx::f32x2_to_e4m3x2(__fmul_rn(__uint_as_float(w[i] << 16), inv),
                                                            __fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), inv));
                            const uint2 q8 = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
                            *reinterpret_cast<uint2*>(stg + r * 128 + ((((chunk >> 1) ^ (r & 7))) << 4) + (chunk & 1) * 8) = q8;
                            if (!bad) *reinterpret_cast<uint2*>(dst + static_cast<size_t>(row0 + pos) * D + chunk * 8) = q8;
                        }
                    } else {
                        uint8_t* stg = stages + s * S::kStageB + (is_v ? S::kTileB : 0) + (chunk >> 3) * S::kHalfBytes;
                        for (int pos = lo; pos < hi_l; ++pos) {
                            const int t = pos - seg_prior, r = pos - tile0;
                            const uint4 val = (t == 0) ? new_row0
                                                       : __ldg(reinterpret_cast<const uint4*>(src + t * (D * 2) + chunk * 16));
                            *reinterpret_cast<uint4*>(stg + r * 128 + (((chunk & 7) ^ (r & 7)) << 4)) = val;
                            if (!bad) *reinterpret_cast<uint4*>(dst + static_cast<size_t>(row0 + pos) * (D * 2) + chunk * 16) = val;
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                }
            }

            if (tile0 + KT > extent) {
                // Clear V rows at or past the unit's last visible key (slots past
                // lens may hold NaN; their probabilities are 0 but 0 * NaN is NaN).
                const int vr0 = extent - tile0;
                const int per_half = (KT - vr0) * 8;
                uint8_t* vbase = stages + s * S::kStageB + S::kTileB;
                const int t0 = S::kTilePar ? lane : tid;
                const int step = S::kTilePar ? 32 : S::kCT;
                for (int idx = t0; idx < (F8 ? 1 : D / 64) * per_half; idx += step) {
                    const int hf = idx / per_half, rem = idx - hf * per_half;
                    *reinterpret_cast<uint4*>(vbase + hf * S::kHalfBytes + (vr0 + (rem >> 3)) * 128 + (rem & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                ptx::fence_proxy_async_smem();
                if (S::kTilePar) __syncwarp(); else ptx::named_barrier_sync(1, S::kCT);
            }
            if (tile0 <= min_lo) {
                // Clear V rows outside every row's window as well (a stale slot
                // must never meet p = 0).
                const int vr1 = min(KT, min_lo - tile0 + 1);
                const int per_half = vr1 * 8;
                uint8_t* vbase = stages + s * S::kStageB + S::kTileB;
                const int t0 = S::kTilePar ? lane : tid;
                const int step = S::kTilePar ? 32 : S::kCT;
                for (int idx = t0; idx < (F8 ? 1 : D / 64) * per_half; idx += step) {
                    const int hf = idx / per_half, rem = idx - hf * per_half;
                    *reinterpret_cast<uint4*>(vbase + hf * S::kHalfBytes + (rem >> 3) * 128 + (rem & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                ptx::fence_proxy_async_smem();
                if (S::kTilePar) __syncwarp(); else ptx::named_barrier_sync(1, S::kCT);
            }
            for (int pass = 0; pass < KW / KWP; ++pass) {
                const int kp = koff + pass * KWP;  // this pass's first key within the tile
                // With a draft tree only tiles wholly before the chunk are free of the mask.
                const int kpass0 = tile0 + kp;  // first key position of this pass
                const bool full_tile = (kpass0 + KWP - 1 <= min_lim) && (kpass0 > max_lo) &&
                                       (!TREE || kpass0 + KWP <= seg_prior);

                // S = Q K^T for this warp's 16 rows x KW keys.
                float sc[NBS][4];
    #pragma unroll
                for (int nb = 0; nb < NBS; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
                if constexpr (F8) {
                    // Key n-block nb: this thread's key is kp + 8*nb + lane/4, and
                    // its 32 bytes d = 32*quad .. 32*quad + 31 (two swizzled 16-byte
                    // chunks) hold k-step kk's four values at bytes 4*kk .. 4*kk + 3.
    #pragma unroll
                    for (int nb = 0; nb < NBS; ++nb) {
                        const int key = kp + nb * 8 + (lane >> 2);
                        const uint32_t row = sK + key * 128;
                        const uint4 u0 = ptx::ld_shared_v4(row + (((2 * quad) ^ (key & 7)) << 4));
                        const uint4 u1 = ptx::ld_shared_v4(row + (((2 * quad + 1) ^ (key & 7)) << 4));
                        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    #pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            uint32_t b0, b1;
                            ptx::e4m3x4_to_f16x2x2(w[kk], b0, b1);
                            ptx::mma_f16_16816(sc[nb], qa[kk], b0, b1);
                        }
                    }
                } else {
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
    #pragma unroll
                        for (int kb = 0; kb < KB; ++kb) {
                            const int mi = lane >> 3;
                            const int key = kp + kb * 16 + (mi >> 1) * 8 + (lane & 7);
                            const int chunk = 2 * kk + (mi & 1);
                            const uint32_t addr = sK + (chunk >> 3) * S::kHalfBytes + key * 128 + (((chunk & 7) ^ (key & 7)) << 4);
                            uint32_t b0, b1, b2, b3;
                            ptx::ldmatrix_x4(addr, b0, b1, b2, b3);
                            ptx::mma_bf16_16816(sc[2 * kb], qa[kk], b0, b1);
                            ptx::mma_bf16_16816(sc[2 * kb + 1], qa[kk], b2, b3);
                        }
                    }
                }

                // Mask (diagonal / ragged tiles only) and online softmax in base 2.
                // The row maximum is taken on the raw scores (the scale is
                // positive) and the scale is folded into the exponent's FMA.  The
                // reference used for the exponentials only moves when a row's
                // maximum passes it by more than kLazyRescale (a factor 2^8 at
                // most on p), and only then are O and l rescaled; O, l and the
                // stored m share that reference, so the result is exact.
                const int kbase = tile0 + kp + 2 * quad;
                float mx0 = -INFINITY, mx1 = -INFINITY;
    #pragma unroll
                for (int nb = 0; nb < NBS; ++nb) {
                    if (!full_tile) {
    #pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int key = kbase + nb * 8 + (e & 1);
                            const int lim = (e < 2) ? lim0 : lim1;
                            if (key > lim || key <= ((e < 2) ? lo0 : lo1)) sc[nb][e] = -INFINITY;
                            else if (TREE && key >= seg_prior &&
                                     !((p.anc[b * p.T + (lim - seg_prior)] >> (key - seg_prior)) & 1ull))
                                sc[nb][e] = -INFINITY;  // a draft token off this query's path to the root
                        }
                    }
                    mx0 = fmaxf(mx0, fmaxf(sc[nb][0], sc[nb][1]));
                    mx1 = fmaxf(mx1, fmaxf(sc[nb][2], sc[nb][3]));
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                mx0 *= sl2;  // -inf stays -inf
                mx1 *= sl2;
                const bool mv0 = mx0 > m0 + kLazyRescale, mv1 = mx1 > m1 + kLazyRescale;
                if (mv0 || mv1) {
                    const float n0 = mv0 ? mx0 : m0, n1 = mv1 ? mx1 : m1;
                    const float al0 = (m0 == -INFINITY) ? 0.f : ptx::ex2(m0 - n0);
                    const float al1 = (m1 == -INFINITY) ? 0.f : ptx::ex2(m1 - n1);
                    l0 *= al0;
                    l1 *= al1;
    #pragma unroll
                    for (int nb = 0; nb < D / 8; ++nb) {
                        o[nb][0] *= al0;
                        o[nb][1] *= al0;
                        o[nb][2] *= al1;
                        o[nb][3] *= al1;
                    }
                    m0 = n0;
                    m1 = n1;
                }
                const float nmu0 = (m0 == -INFINITY) ? 0.f : -m0;
                const float nmu1 = (m1 == -INFINITY) ? 0.f : -m1;
                float ps0 = 0.f, ps1 = 0.f;
    #pragma unroll
                for (int nb = 0; nb < NBS; ++nb) {
                    sc[nb][0] = ptx::ex2(fmaf(sc[nb][0], sl2, nmu0));
                    sc[nb][1] = ptx::ex2(fmaf(sc[nb][1], sl2, nmu0));
                    sc[nb][2] = ptx::ex2(fmaf(sc[nb][2], sl2, nmu1));
                    sc[nb][3] = ptx::ex2(fmaf(sc[nb][3], sl2, nmu1));
                    ps0 += sc[nb][0] + sc[nb][1];
                    ps1 += sc[nb][2] + sc[nb][3];
                }
                l0 += ps0;
                l1 += ps1;

                // O += P V.
    #pragma unroll
                for (int kb = 0; kb < KB && F8; ++kb) {
                    // P (f16) x V (E4M3 -> f16).  Output n-block jd, column
                    // lane/4 = g stands for d = 16*g + jd, so this thread reads one
                    // 16-byte chunk (g) of each of its four key rows, and the two
                    // keys of a B register pair come from two rows (byte permute).
                    uint32_t a[4];
                    a[0] = ptx::pack_f16x2(sc[2 * kb][0], sc[2 * kb][1]);
                    a[1] = ptx::pack_f16x2(sc[2 * kb][2], sc[2 * kb][3]);
                    a[2] = ptx::pack_f16x2(sc[2 * kb + 1][0], sc[2 * kb + 1][1]);
                    a[3] = ptx::pack_f16x2(sc[2 * kb + 1][2], sc[2 * kb + 1][3]);
                    const int k0 = kp + kb * 16 + 2 * quad, g = lane >> 2;
                    auto vrow = [&](int k) { return ptx::ld_shared_v4(sV + k * 128 + ((g ^ (k & 7)) << 4)); };
                    const uint4 r0 = vrow(k0), r1 = vrow(k0 + 1), r8 = vrow(k0 + 8), r9 = vrow(k0 + 9);
                    const uint32_t x0[4] = {r0.x, r0.y, r0.z, r0.w}, x1[4] = {r1.x, r1.y, r1.z, r1.w};
                    const uint32_t x8[4] = {r8.x, r8.y, r8.z, r8.w}, x9[4] = {r9.x, r9.y, r9.z, r9.w};
    #pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t b0[4], b1[4];  // n-blocks 4i .. 4i+3: keys (k0, k0+1) and (k0+8, k0+9)
                        ptx::e4m3x4_to_f16x2x2(ptx::prmt(x0[i], x1[i], 0x5140), b0[0], b0[1]);
                        ptx::e4m3x4_to_f16x2x2(ptx::prmt(x0[i], x1[i], 0x7362), b0[2], b0[3]);
                        ptx::e4m3x4_to_f16x2x2(ptx::prmt(x8[i], x9[i], 0x5140), b1[0], b1[1]);
                        ptx::e4m3x4_to_f16x2x2(ptx::prmt(x8[i], x9[i], 0x7362), b1[2], b1[3]);
    #pragma unroll
                        for (int m = 0; m < 4; ++m) ptx::mma_f16_16816(o[4 * i + m], a, b0[m], b1[m]);
                    }
                }
    #pragma unroll
                for (int kb = 0; kb < KB && !F8; ++kb) {
                    uint32_t a[4];
                    a[0] = ptx::pack_bf16x2(sc[2 * kb][0], sc[2 * kb][1]);
                    a[1] = ptx::pack_bf16x2(sc[2 * kb][2], sc[2 * kb][3]);
                    a[2] = ptx::pack_bf16x2(sc[2 * kb + 1][0], sc[2 * kb + 1][1]);
                    a[3] = ptx::pack_bf16x2(sc[2 * kb + 1][2], sc[2 * kb + 1][3]);
    #pragma unroll
                    for (int dc = 0; dc < D / 16; ++dc) {
                        const int mi = lane >> 3;
                        const int key = kp + kb * 16 + (mi & 1) * 8 + (lane & 7);
                        const int chunk = 2 * dc + (mi >> 1);
                        const uint32_t addr = sV + (chunk >> 3) * S::kHalfBytes + key * 128 + (((chunk & 7) ^ (key & 7)) << 4);
                        uint32_t b0, b1, b2, b3;
                        ptx::ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                        ptx::mma_bf16_16816(o[2 * dc], a, b0, b1);
                        ptx::mma_bf16_16816(o[2 * dc + 1], a, b2, b3);
                    }
                }
            }

            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar0 + 8 * (kStages + s));
        }

        const bool seg_end = (x == x1 - 1) || (j == nt - 1);
        if (seg_end) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            if (NM > 1) {
                // Merge the NM softmax states of each m-tile into its ms == 0 warp.
                const int r0 = lane >> 2;
                if (quad == 0) {
                    ml[(warp * 16 + r0) * 2 + 0] = m0;
                    ml[(warp * 16 + r0) * 2 + 1] = l0;
                    ml[(warp * 16 + r0 + 8) * 2 + 0] = m1;
                    ml[(warp * 16 + r0 + 8) * 2 + 1] = l1;
                }
                ptx::named_barrier_sync(1, S::kCT);
                float mf0 = -INFINITY, mf1 = -INFINITY;
#pragma unroll
                for (int k2 = 0; k2 < NM; ++k2) {
                    const int w2 = S::kTilePar ? k2 : mt + k2 * MT;
                    mf0 = fmaxf(mf0, ml[(w2 * 16 + r0) * 2]);
                    mf1 = fmaxf(mf1, ml[(w2 * 16 + r0 + 8) * 2]);
                }
                const float mfu0 = (mf0 == -INFINITY) ? 0.f : mf0;
                const float mfu1 = (mf1 == -INFINITY) ? 0.f : mf1;
                float lf0 = 0.f, lf1 = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < NM; ++k2) {
                    const int w2 = S::kTilePar ? k2 : mt + k2 * MT;
                    lf0 += ml[(w2 * 16 + r0) * 2 + 1] * ptx::ex2(ml[(w2 * 16 + r0) * 2] - mfu0);
                    lf1 += ml[(w2 * 16 + r0 + 8) * 2 + 1] * ptx::ex2(ml[(w2 * 16 + r0 + 8) * 2] - mfu1);
                }
                const float f0 = ptx::ex2(m0 - mfu0), f1 = ptx::ex2(m1 - mfu1);
#pragma unroll
                for (int nb = 0; nb < D / 8; ++nb) {
                    o[nb][0] *= f0;
                    o[nb][1] *= f0;
                    o[nb][2] *= f1;
                    o[nb][3] *= f1;
                }
                if (ms > 0) {
                    float* ob = obuf + ((ms - 1) * MT + mt) * 16 * D;
#pragma unroll
                    for (int nb = 0; nb < D / 8; ++nb) {
                        const int col = nb * 8 + 2 * quad;
                        *reinterpret_cast<float2*>(ob + r0 * D + col) = make_float2(o[nb][0], o[nb][1]);
                        *reinterpret_cast<float2*>(ob + (r0 + 8) * D + col) = make_float2(o[nb][2], o[nb][3]);
                    }
                }
                ptx::named_barrier_sync(1, S::kCT);
                if (ms == 0) {
#pragma unroll
                    for (int k2 = 1; k2 < NM; ++k2) {
                        const float* ob = obuf + ((k2 - 1) * MT + mt) * 16 * D;
#pragma unroll
                        for (int nb = 0; nb < D / 8; ++nb) {
                            const int col = nb * 8 + 2 * quad;
                            const float2 a = *reinterpret_cast<const float2*>(ob + r0 * D + col);
                            const float2 c = *reinterpret_cast<const float2*>(ob + (r0 + 8) * D + col);
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
                ptx::named_barrier_sync(1, S::kCT);
            }

            // Writers: in the shared-merge layout the ms == 0 warp of each
            // m-tile; with warps owning whole tiles, every warp that took at
            // least one tile of this unit segment.  The unit's output is written
            // here when this writer saw all of it (the whole unit ran in this
            // CTA, and with warps owning tiles, the unit is a single tile);
            // otherwise a partial (m, l, O) goes to sub-slot (u + CTA) * ways +
            // warp for the combine kernel.
            const bool writer = S::kTilePar ? (seg_tiles > 0) : (ms == 0);
            const bool sole = (seg_j0 == 0) && (j == nt - 1) && (!S::kTilePar || nt == 1);
            if (writer) {
                const int slot = (cur.q * p.Hkv + kvh + blockIdx.x) * S::kWays + (S::kTilePar ? warp : 0);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int lim = h ? lim1 : lim0;
                    if (lim < 0) continue;  // padding row or padded query: never written here
                    const float l = h ? l1 : l0;
                    if (sole) {
                        // The whole unit ran in this CTA: normalise and write the output.
                        const int r = rb * RPB + lrow0 + 8 * h;
                        const int g = r / p.T, t = r % p.T;
                        const float inv = l > 0.f ? (F8 ? p.vscale[kvh] : 1.f) / l : 0.f;
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                                             ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * p.T + t) * D;
                        if constexpr (F8) {
                            // o[jd][2h] is d = 32*quad + jd, o[jd][2h+1] is d = 32*quad + 16 + jd
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                uint32_t w[8];
#pragma unroll
                                for (int m = 0; m < 8; ++m)
                                    w[m] = ptx::pack_bf16x2(o[2 * m][2 * h + half] * inv, o[2 * m + 1][2 * h + half] * inv);
                                uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * quad + 16 * half);
                                d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                                d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
                            }
                        } else {
#pragma unroll
                            for (int nb = 0; nb < D / 8; ++nb) {
                                const int col = nb * 8 + 2 * quad;
                                *reinterpret_cast<uint32_t*>(dst + col) =
                                    ptx::pack_bf16x2(o[nb][2 * h] * inv, o[nb][2 * h + 1] * inv);
                            }
                        }
                    } else {
                        // Part of a unit seen by several writers: leave (m, l, O)
                        // for the combine kernel.
                        float* part = p.partials + (static_cast<size_t>(slot) * p.part_rows + lrow0 + 8 * h) * PS;
                        if constexpr (F8) {
                            // natural column order, V scale applied (the merge is linear in O)
                            const float vs = p.vscale[kvh];
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                float4* d4 = reinterpret_cast<float4*>(part + 32 * quad + 16 * half);
#pragma unroll
                                for (int m = 0; m < 4; ++m)
                                    d4[m] = make_float4(o[4 * m][2 * h + half] * vs, o[4 * m + 1][2 * h + half] * vs,
                                                        o[4 * m + 2][2 * h + half] * vs, o[4 * m + 3][2 * h + half] * vs);
                            }
                        } else {
#pragma unroll
                            for (int nb = 0; nb < D / 8; ++nb) {
                                const int col = nb * 8 + 2 * quad;
                                *reinterpret_cast<float2*>(part + col) = make_float2(o[nb][2 * h], o[nb][2 * h + 1]);
                            }
                        }
                        if (quad == 0) {
                            part[D] = h ? m1 : m0;
                            part[D + 1] = l;
                        }
                    }
                }
            }
        }
        cur.advance(wp);
    }
}

// One CTA per unit.  Units written in full by the attention kernel return at
// once; for the others, the log-sum-exp merge of the partials (m_i, l_i, O_i)
// of every writer, o = sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i with
// M = max_i m_i, is written for the unit's valid rows.  Writers: CTAs c0..c1
// (those whose tile ranges meet the unit) and, when warps own whole tiles,
// each warp w of such a CTA that took one of the unit's tiles (tile k of the
// CTA's range goes to warp k mod ways).
constexpr int kCombineThreads = 128;
constexpr int kCombineChunk = 8;   // partials loaded together (independent loads)

// The partition as the combine kernel sees it: host plan in the parameters
// (parameter space) or the device plan.
template <bool DP>
struct CPart;
template <>
struct CPart<false> {
    const CombineParams& p;
    __device__ __forceinline__ int gstart(int i) const { return p.gstart[i]; }
    __device__ __forceinline__ int cta_start(int i) const { return p.cta_start[i]; }
    __device__ __forceinline__ int n_new(int b) const { return p.n_new[b]; }
};
template <>
struct CPart<true> {
    const CombineParams& p;
    const int* cta_start_sh;  // the plan's CTA starts, staged in shared memory (searched per thread)
    __device__ __forceinline__ int gstart(int i) const { return p.dplan->gstart[i]; }
    __device__ __forceinline__ int cta_start(int i) const { return cta_start_sh[i]; }
    __device__ __forceinline__ int n_new(int b) const { return p.dplan->n_new[b]; }
};

template <bool DP>
__device__ __forceinline__ CPart<DP> make_cpart(const CombineParams& p, const int* sh);
template <>
__device__ __forceinline__ CPart<false> make_cpart<false>(const CombineParams& p, const int*) {
    return CPart<false>{p};
}
template <>
__device__ __forceinline__ CPart<true> make_cpart<true>(const CombineParams& p, const int* sh) {
    return CPart<true>{p, sh};
}

// CTA whose tile range holds tile x: largest i with cta_start[i] <= x (CTAs
// with empty ranges repeat the next start, so the owner is the last of them).
template <bool DP>
__device__ __forceinline__ int cta_holding(const CPart<DP>& w, int num_ctas, long long x) {
    int lo = 0, hi = num_ctas - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (w.cta_start(mid) <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <bool DP, int D>
__global__ void __launch_bounds__(kCombineThreads) combine_bf16_kernel(const __grid_constant__ CombineParams p) {
    constexpr int PS = part_stride(D);
    constexpr int C4 = D / 4;  // 4-column slices of a row
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    if (DP && p.dplan->skip) return;
    // A device plan lives in global memory: stage its CTA starts in shared
    // memory once (one parallel round trip) instead of searching them there.
    __shared__ int cta_start_sh[DP ? kMaxCtas + 1 : 1];
    if constexpr (DP) {
        for (int i = threadIdx.x; i <= p.num_ctas; i += kCombineThreads) cta_start_sh[i] = p.dplan->cta_start[i];
        __syncthreads();
    }
    const CPart<DP> cw = make_cpart<DP>(p, cta_start_sh);
    const int u = blockIdx.x;
    const int q = u / p.Hkv, kvh = u - q * p.Hkv;
    const int nt = (cw.gstart(q + 1) - cw.gstart(q)) / p.Hkv;
    if (nt == 0) return;
    const int us = cw.gstart(q) + kvh * nt, ue = us + nt - 1;
    const int c0 = cta_holding(cw, p.num_ctas, us), c1 = cta_holding(cw, p.num_ctas, ue);
    if (c0 == c1 && (p.ways == 1 || nt == 1)) return;  // written by the attention kernel
    const int ncand = (c1 - c0 + 1) * p.ways;
    const int b = q / p.RB, rb = q - b * p.RB;
    const int nn = cw.n_new(b);
    for (int idx = threadIdx.x; idx < p.part_rows * C4; idx += kCombineThreads) {
        const int lr = idx / C4, c4 = idx % C4;
        const int r = rb * p.RPB + lr;
        if (r >= p.R || (r % p.T) >= nn) continue;
        const float* base = p.partials + ((static_cast<size_t>(u + c0) * p.ways) * p.part_rows + lr) * PS;
        const size_t stride = static_cast<size_t>(p.part_rows) * PS;  // next sub-slot
        // One pass, merging chunks of partials online: (m, l, acc) <- merge.
        float m = -INFINITY, l = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int e0 = 0; e0 < ncand; e0 += kCombineChunk) {
            float mi[kCombineChunk], li[kCombineChunk];
            float4 oi[kCombineChunk];
#pragma unroll
            for (int k = 0; k < kCombineChunk; ++k) {
                // Candidate e = (CTA c0 + e / ways, warp e % ways): did it write?
                const int e = e0 + k;
                bool valid = e < ncand;
                if (valid) {
                    const int ci = e / p.ways, w = e - ci * p.ways;
                    const int x0 = cw.cta_start(c0 + ci), x1 = cw.cta_start(c0 + ci + 1);
                    const int la = max(us, x0) - x0, lb = min(ue, x1 - 1) - x0;
                    valid = (lb - la + 1 >= p.ways) || ((w - la % p.ways + p.ways) % p.ways <= lb - la);
                }
                const float* part = base + (valid ? e : 0) * stride;
                mi[k] = valid ? part[D] : -INFINITY;
                li[k] = valid ? part[D + 1] : 0.f;
                oi[k] = valid ? reinterpret_cast<const float4*>(part)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < kCombineChunk; ++k) {
                const float mn = fmaxf(m, mi[k]);
                if (mn == -INFINITY) continue;
                const float a = ptx::ex2(m - mn), c = ptx::ex2(mi[k] - mn);
                l = l * a + li[k] * c;
                acc.x = acc.x * a + oi[k].x * c;
                acc.y = acc.y * a + oi[k].y * c;
                acc.z = acc.z * a + oi[k].z * c;
                acc.w = acc.w * a + oi[k].w * c;
                m = mn;
            }
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int g = r / p.T, t = r % p.T;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                             ((static_cast<size_t>(b) * p.Hq + kvh * p.G + g) * p.T + t) * D + c4 * 4;
        store_bf16x4(dst, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// Plan of one device-resident step (one CTA of 1024 threads): check every
// row (0 <= n_new <= T, lens + n_new <= max_len; a bad row rejects the whole
// step, nothing is written and the error word records it), then the same work
// partition the host planner builds (per-group tile starts, per-CTA tile
// starts) from the device lengths, and finally advance the lengths.
constexpr int kPlanThreads = 1024;
__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const __grid_constant__ PlanParams p) {
    ptx::grid_dependency_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    DevicePlan* plan = p.plan;
    int bad = 0;
    for (int b = tid; b < p.B; b += kPlanThreads) {
        const int L = p.lens[b], n = p.n_new[b];
        const bool room = p.ring ? (n <= p.max_len - p.window + 1 && L <= 0x7fffffff - p.max_len - n)
                                 : (L <= p.max_len - n);
        bad |= (L < 0 || n < 0 || n > p.T || !room) ? 1 : 0;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            plan->skip = 1;
            plan->total_tiles = 0;
            atomicExch(p.err, kDevOverflow);
        }
        ptx::launch_dependents();
        return;
    }
    for (int b = tid; b < p.B; b += kPlanThreads) {
        plan->prior[b] = p.lens[b];
        plan->n_new[b] = p.n_new[b];
    }
    // Tiles of group q = b * RB + rb: Hkv units over the key tiles from the
    // window of the block's earliest query to one past its largest visible key.
    int tiles = 0, ft = 0;
    if (tid < p.NB) {
        const int b = tid / p.RB, rb = tid - b * p.RB;
        const int prior = p.lens[b], n = p.n_new[b];
        const int r0 = rb * p.RPB, r1 = min(p.R, r0 + p.RPB);
        int extent = 0, qmin = 0x7fffffff;
        if (r1 - r0 >= p.T) {
            if (n > 0) {
                extent = prior + min(p.T, n);
                qmin = prior;
            }
        } else {
            for (int r = r0; r < r1; ++r) {
                const int t = r % p.T;
                if (t < n) {
                    extent = max(extent, prior + t + 1);
                    qmin = min(qmin, prior + t);
                }
            }
        }
        const int kfirst = (extent > 0 && p.window > 0) ? max(0, qmin - p.window + 1) : 0;
        ft = kfirst / p.key_tile;
        tiles = extent > 0 ? ((extent - 1) / p.key_tile + 1 - ft) * p.Hkv : 0;
    }
    // Block-wide exclusive scan of the group tile counts.
    __shared__ int warp_sum[kPlanThreads / 32];
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - tiles + (warp > 0 ? warp_sum[warp - 1] : 0);
    const int total = warp_sum[kPlanThreads / 32 - 1];
    if (tid < p.NB) plan->gstart[tid] = excl;
    if (tid == 0) {
        plan->gstart[p.NB] = total;
        plan->total_tiles = total;
        plan->skip = 0;
    }
    for (int i = tid; i <= p.num_ctas; i += kPlanThreads)
        plan->cta_start[i] = static_cast<int>(static_cast<long long>(i) * total / p.num_ctas);
    __syncthreads();  // every read of lens above is done
    for (int b = tid; b < p.B; b += kPlanThreads) p.lens[b] += p.n_new[b];
    ptx::launch_dependents();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int MT, bool DP, bool TREE, bool F8, int D>
cudaError_t launch_mt(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int grid,
                      cudaStream_t stream) {
    using S = Shape<MT, F8, D>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_splitkv_bf16_kernel<MT, DP, TREE, F8, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(S::kSmem));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaError_t e = launch_pdl(decode_splitkv_bf16_kernel<MT, DP, TREE, F8, D>, dim3(grid), dim3(S::kThreads),
                               S::kSmem, stream, p, tmK, tmV);
    if (e != cudaSuccess) return e;
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

template <bool F8, int D>
DecodeLaunch launch_shape_t(int mt) {
    switch (mt) {
        case 1: return DecodeLaunch{1, Shape<1, F8, D>::kThreads, Shape<1, F8, D>::kSmem, Shape<1, F8, D>::kWays};
        case 2: return DecodeLaunch{2, Shape<2, F8, D>::kThreads, Shape<2, F8, D>::kSmem, Shape<2, F8, D>::kWays};
        default: return DecodeLaunch{4, Shape<4, F8, D>::kThreads, Shape<4, F8, D>::kSmem, Shape<4, F8, D>::kWays};
    }
}

DecodeLaunch decode_launch_shape(int mt, bool fp8, int d) {
    if (fp8) return launch_shape_t<true, 128>(mt);
    return d == 64 ? launch_shape_t<false, 64>(mt) : launch_shape_t<false, 128>(mt);
}

template <bool F8, int D>
cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int mt, int grid,
                            cudaStream_t stream) {
    if (p.dplan)
        return (mt == 1 && !p.anc) ? launch_mt<1, true, false, F8, D>(p, tmK, tmV, grid, stream) : cudaErrorInvalidValue;
    if (p.anc) {
        switch (mt) {
            case 1: return launch_mt<1, false, true, F8, D>(p, tmK, tmV, grid, stream);
            case 2: return launch_mt<2, false, true, F8, D>(p, tmK, tmV, grid, stream);
            case 4: return launch_mt<4, false, true, F8, D>(p, tmK, tmV, grid, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (mt) {
        case 1: return launch_mt<1, false, false, F8, D>(p, tmK, tmV, grid, stream);
        case 2: return launch_mt<2, false, false, F8, D>(p, tmK, tmV, grid, stream);
        case 4: return launch_mt<4, false, false, F8, D>(p, tmK, tmV, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int mt,
                               int grid, bool fp8, int d, cudaStream_t stream) {
    if (fp8) return d == 128 ? launch_decode_t<true, 128>(p, tmK, tmV, mt, grid, stream) : cudaErrorInvalidValue;
    if (d == 64) return launch_decode_t<false, 64>(p, tmK, tmV, mt, grid, stream);
    return d == 128 ? launch_decode_t<false, 128>(p, tmK, tmV, mt, grid, stream) : cudaErrorInvalidValue;
}

cudaError_t launch_combine_bf16(const CombineParams& p, cudaStream_t stream) {
    if (p.d != 64 && p.d != 128) return cudaErrorInvalidValue;
    auto k = p.dplan ? (p.d == 64 ? combine_bf16_kernel<true, 64> : combine_bf16_kernel<true, 128>)
                     : (p.d == 64 ? combine_bf16_kernel<false, 64> : combine_bf16_kernel<false, 128>);
    cudaError_t e = launch_pdl(k, dim3(p.NB * p.Hkv), dim3(kCombineThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_decode_plan(const PlanParams& p, cudaStream_t stream) {
    cudaError_t e = launch_pdl(decode_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace kvc
