// Host side of libkvc: the C ABI declared in kvc.h.
//
// Holds per-layer, per-row lengths (host-authoritative), validates every
// argument before anything is enqueued (so an error changes nothing), plans
// the split-KV work partition from the host lengths without a device sync,
// and launches the kernels on the caller's stream.
//
// Cache semantics follow "Implement grouped-query attention over a
// preallocated KV cache..." ("A strong answer": KVCache.append raises past
// max_len, lengths grow after the write) and "16. Prefill, decode and the KV
// cache" ("Layout and validity": per-layer lengths, length refusing when a
// forward pass stopped part-way, truncate, reset).

#include <math.h>

#include <cmath>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "kvc_internal.h"

using namespace kvc;

struct kvc_cache {
    int layers = 0, B = 0, Hkv = 0, max_len = 0, d = 0;
    kvc_dtype dtype = KVC_F32;
    int esize = 4;  // bytes a stored value
    // FP8 E4M3 caches: K and V scale of every (layer, KV head), [layers * Hkv]
    std::vector<float> kscale, vscale;
    std::vector<void*> k, v;
    std::vector<int64_t> lens;  // [layers * B]
    // device state, set up on first launch
    bool dev_ready = false;
    int device = -1;
    int num_sms = 0;
    std::vector<CUtensorMap> tmK, tmV;        // 64-row boxes (split-KV kernel)
    std::vector<CUtensorMap> tmK128, tmV128;  // 128-row boxes (prefill kernel)
    std::vector<char> tm_ready;
    const void* last_ws = nullptr;
    uint64_t launches = 0;  // kernels this handle has enqueued
    // Device-resident lengths (caller-owned int32 [layers][B]) while a run of
    // graph-capturable steps owns them; the host copy is stale meanwhile.
    int32_t* dev_lens = nullptr;
    bool lens_on_device = false;
    // Sliding window (0 = none) and ring storage (slot = position mod max_len).
    int window = 0;
    bool ring = false;
    // Paged storage (table set): buffers [num_pages, Hkv, page, d], a device
    // block table [B, mpr]; max_len is the logical capacity mpr * page.
    Paging pg{nullptr, 0, 0, 0};
    // Host-buffer calls (kvc_append_attention_host): two device staging slots
    // (q, k_new, v_new, out of one call each) used in turn, the two copy
    // streams (inputs in, outputs out) and each slot's events.
    struct HostSlot {
        void* buf = nullptr;
        size_t bytes = 0;
        cudaEvent_t in_ready = nullptr, computed = nullptr, out_done = nullptr;
    };
    HostSlot hslot[2];
    int hnext = 0;
    cudaStream_t h2d = nullptr, d2h = nullptr;
};

namespace {

// Query rows per KV head (G * T) above which attention runs on the tcgen05
// kernel; at or below it, on the split-KV kernel (mma.sync, appends fused).
// Measured on the verify shape (B = 64, S = 4096): bf16 at 8 rows, the
// split-KV kernel is ahead by about 2 %, at 16 rows the tcgen05 kernel by
// about 3 %.  An FP8 cache converts its tiles in shared memory on the tcgen05
// kernel, so there the split-KV kernel (128-key FP8 tiles) leads up to 32
// rows (2,855 against 2,484 GB/s at 32) and the tcgen05 kernel from 64 (2,524
// against 1,670).
constexpr int kTcMinRows = 12;
constexpr int kTcMinRowsFp8 = 32;
int tc_min_rows(const kvc_cache* c) { return c->dtype == KVC_FP8_E4M3 ? kTcMinRowsFp8 : kTcMinRows; }
// Caches served by the generic kernel (attn_f32.cu) only: fp32 storage, and
// bf16 or FP8 storage whose head dimension has no TMA kernel (the split-KV
// kernel takes d = 128, and d = 64 for bf16; the tensor-core kernel d = 128).
bool generic_path(const kvc_cache* c) {
    return c->dtype == KVC_F32 || !(c->d == kHeadDimBf16 || (c->d == kHeadDimSmall && c->dtype == KVC_BF16));
}
// Head dimension the tensor-core kernel is built for.
bool tc_capable(const kvc_cache* c) { return !generic_path(c) && c->d == kHeadDimBf16; }
// Calls with more query rows per KV head than the split-KV kernel's 64 on a
// cache the tensor-core kernel cannot take (bf16, d = 64) run on the generic kernel.
bool generic_call(const kvc_cache* c, int R) { return generic_path(c) || (!tc_capable(c) && R > 64); }
constexpr int kTcMaxLen = 0xFFFF * 128;  // key tiles of a piece are packed in 16 bits

thread_local std::string g_last_error;

kvc_status fail(kvc_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kvc_status fail(kvc_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

kvc_status ok() { return KVC_OK; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvc_status cuda_fail(cudaError_t e, const char* what) {
    return fail(KVC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {  // looked up once, thread-safe
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// The device this process's handles run on: the kernels' shared-memory
// attributes are set once, for the first device that launches them.
std::atomic<int> g_device{-1};

// Bind the handle to the current device on its first launch; afterwards every
// launching call must find that device current (its buffers live there).
kvc_status ensure_device(kvc_cache* c) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (c->dev_ready) {
        if (dev != c->device) return fail(KVC_ERR_ARG, "current device %d is not the cache's device %d", dev, c->device);
        return ok();
    }
    int bound = -1;
    if (!g_device.compare_exchange_strong(bound, dev) && bound != dev)
        return fail(KVC_ERR_ARG, "the library serves one device per process (device %d; current device %d)", bound, dev);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    c->device = dev;
    c->num_sms = sms;
    c->dev_ready = true;
    return ok();
}

// 2-D view [rows, 128 values] with boxes of box_rows rows x 128 bytes (64
// bf16 columns, or all 128 one-byte E4M3 columns) and the 128-byte swizzle.
kvc_status encode_rows_map(CUtensorMap* m, const void* base, cuuint64_t rows, cuuint32_t box_rows, bool fp8 = false,
                           int d = kHeadDimBf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * (fp8 ? 1 : 2)};
    cuuint32_t box[2] = {fp8 ? 128u : 64u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                    dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return ok();
}

// One layer's K and V as rows = B*Hkv*max_len: 64-row and 128-row boxes.
kvc_status encode_layer_maps(kvc_cache* c, int layer) {
    if (c->tm_ready[layer]) return ok();
    const cuuint64_t rows = c->pg.table ? static_cast<cuuint64_t>(c->pg.num_pages) * c->Hkv * c->pg.page
                                        : static_cast<cuuint64_t>(c->B) * c->Hkv * c->max_len;
    kvc_status s;
    const bool fp8 = c->dtype == KVC_FP8_E4M3;
    const int kt = key_tile_keys(c->d, fp8);  // the split-KV kernel's tile for this cache
    if ((s = encode_rows_map(&c->tmK[layer], c->k[layer], rows, kt, fp8, c->d))) return s;
    if ((s = encode_rows_map(&c->tmV[layer], c->v[layer], rows, kt, fp8, c->d))) return s;
    if (tc_capable(c)) {
        if ((s = encode_rows_map(&c->tmK128[layer], c->k[layer], rows, 128, fp8))) return s;
        if ((s = encode_rows_map(&c->tmV128[layer], c->v[layer], rows, 128, fp8))) return s;
    }
    c->tm_ready[layer] = 1;
    return ok();
}

// ---------------------------------------------------------------------------
// Validation shared by append / attention
// ---------------------------------------------------------------------------

kvc_status check_layer(const kvc_cache* c, int layer) {
    if (!c) return fail(KVC_ERR_ARG, "null cache handle");
    if (layer < 0 || layer >= c->layers) return fail(KVC_ERR_ARG, "layer %d outside 0..%d", layer, c->layers - 1);
    return ok();
}

kvc_status validate_append(const kvc_cache* c, int layer, const void* k_new, const void* v_new, int T,
                           const int32_t* n_new, int* max_n) {
    kvc_status s = check_layer(c, layer);
    if (s) return s;
    if (T < 0) return fail(KVC_ERR_ARG, "T = %d < 0", T);
    if (c->B > 0 && !n_new) return fail(KVC_ERR_ARG, "n_new is null");
    const int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    int mx = 0;
    for (int b = 0; b < c->B; ++b) {
        if (n_new[b] < 0 || n_new[b] > T)
            return fail(KVC_ERR_SHAPE, "row %d: n_new = %d outside 0..%d", b, n_new[b], T);
        mx = std::max(mx, static_cast<int>(n_new[b]));
    }
    for (int b = 0; b < c->B; ++b) {
        if (c->ring) {
            // A ring chunk must fit beside its window: its first query still
            // needs the window - 1 keys before it.
            if (n_new[b] > c->max_len - c->window + 1)
                return fail(KVC_ERR_OVERFLOW, "row %d: a ring chunk of %d tokens does not fit beside a window of %d in %d slots",
                            b, n_new[b], c->window, c->max_len);
            if (lens[b] + n_new[b] > 0x7fffffffll - c->max_len)
                return fail(KVC_ERR_OVERFLOW, "row %d: position count past the int32 range", b);
        } else if (lens[b] + n_new[b] > c->max_len) {
            return fail(KVC_ERR_OVERFLOW, "row %d: %lld tokens > max_len %d", b,
                        static_cast<long long>(lens[b] + n_new[b]), c->max_len);
        }
    }
    if (mx > 0) {
        if (!k_new || !v_new) return fail(KVC_ERR_ARG, "k_new / v_new is null");
        if (!aligned16(k_new) || !aligned16(v_new)) return fail(KVC_ERR_ARG, "k_new / v_new not 16-byte aligned");
    }
    *max_n = mx;
    return ok();
}

struct AttnPlan {
    bool generic = false;  // the call runs on the generic kernel
    int Hq = 0, G = 0, T = 0, R = 0;
    int mt = 0, RPB = 0, RB = 0, NB = 0, units = 0, ways = 1, part_rows = 0;
    int splits = 1;  // generic kernel: CTAs per (row block, KV head, row)
    size_t ws_err = 0, ws_plan = 0, ws_partials = 0, ws_total = 0;
    // Least workspace the call runs with: the tensor-core path needs only the
    // header (with less room it cuts fewer items into pieces).
    size_t ws_min = 0;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

kvc_status plan_shape(const kvc_cache* c, int Hq, int T, int num_ctas, AttnPlan* pl) {
    if (Hq <= 0) return fail(KVC_ERR_ARG, "q_heads = %d", Hq);
    if (Hq % c->Hkv != 0) return fail(KVC_ERR_SHAPE, "q_heads %d is not a multiple of kv_heads %d", Hq, c->Hkv);
    if (T < 0) return fail(KVC_ERR_ARG, "T = %d < 0", T);
    pl->Hq = Hq;
    pl->G = Hq / c->Hkv;
    pl->T = T;
    const long long R = static_cast<long long>(pl->G) * T;
    if (R > (1ll << 30)) return fail(KVC_ERR_ARG, "G * T too large");
    pl->R = static_cast<int>(R);
    pl->generic = generic_call(c, pl->R);
    if (!pl->generic) {
        pl->mt = pl->R <= 16 ? 1 : (pl->R <= 32 ? 2 : 4);
        pl->RPB = 16 * pl->mt;
        pl->RB = std::max(1, (pl->R + pl->RPB - 1) / pl->RPB);
        // Only the split-KV kernel works in (row, row block) groups.  A call
        // with more than 64 rows per KV head (more than any tree call takes)
        // always runs on the tensor cores, unless the cache is too long for
        // them; it plans no groups and needs no split-KV partials.
        const bool tc_only = pl->R > 64 && c->max_len <= kTcMaxLen && tc_capable(c);
        const long long NB = tc_only ? 0 : static_cast<long long>(c->B) * pl->RB;
        if (NB > kMaxGroups)
            return fail(KVC_ERR_ARG, "B * ceil(G*T / %d) = %lld exceeds %d row blocks", pl->RPB, NB, kMaxGroups);
        pl->NB = static_cast<int>(NB);
        pl->units = pl->NB * c->Hkv;
        // Layout: the header (error word, merge counters), then the partials of
        // the units that straddle CTAs.  Only the header needs to start at
        // zero; the merge counters return to zero after each use.
        pl->ws_err = kWsHeaderBytes;
        // device-computed plans of resident-length steps, then the ancestor
        // masks of a tree-verify call
        pl->ws_plan = round_up(sizeof(DevicePlan), 256) + round_up(kMaxTreeQueries * sizeof(uint64_t), 256);
        pl->ways = decode_launch_shape(pl->mt, c->dtype == KVC_FP8_E4M3, c->d).ways;
        pl->part_rows = std::min(pl->R, pl->RPB);
        pl->ws_partials = tc_only ? 0
                                  : static_cast<size_t>(pl->units + num_ctas) * pl->ways * pl->part_rows *
                                        (c->d + 4) * sizeof(float);
        pl->ws_min = pl->ws_err + pl->ws_plan + pl->ws_partials;
        if (pl->R > tc_min_rows(c) && tc_capable(c)) {
            // The tensor-core kernel: up to two partial slots (2 row tiles x
            // 128 rows x (d + 4) floats) per SM share boundary.
            const size_t prefill = static_cast<size_t>(2) * std::min(num_ctas, kMaxCtas) * 2 * 128 *
                                   (kHeadDimBf16 + 4) * sizeof(float);
            pl->ws_partials = std::max(pl->ws_partials, prefill);
            if (c->max_len <= kTcMaxLen) pl->ws_min = pl->ws_err + pl->ws_plan;
        }
        pl->ws_total = pl->ws_err + pl->ws_plan + pl->ws_partials;
    } else {
        // Generic kernel: one CTA per (16-row block, KV head, row).  With
        // fewer of those than twice the SMs (decode), each one's key range is
        // split across up to 16 CTAs (at most one a 64-key tile of max_len),
        // about 16 an SM, which leave partials in the workspace; the last to
        // finish merges.
        const long long units = static_cast<long long>((pl->R + 15) / 16) * c->Hkv * c->B;
        if (units > 0 && units < 2ll * num_ctas) {
            const long long want = (16ll * num_ctas + units - 1) / units;  // measured: 4, 8, 16 an SM
            pl->splits = static_cast<int>(std::min<long long>({want, kGenericMaxSplits, (c->max_len + 63) / 64}));
        }
        if (pl->splits > 1) {
            pl->ws_err = kWsHeaderBytes;  // error word, then the per-unit arrival counters
            pl->ws_partials = static_cast<size_t>(units) * pl->splits * 16 * (c->d + 2) * sizeof(float);
            pl->ws_total = pl->ws_min = pl->ws_err + pl->ws_partials;
        }
    }
    return ok();
}

kvc_status validate_attention(const kvc_cache* c, int layer, const void* q, int Hq, int T, const int32_t* n_new,
                              const void* out, const int64_t* lens_after, AttnPlan* pl, int num_ctas) {
    kvc_status s = check_layer(c, layer);
    if (s) return s;
    s = plan_shape(c, Hq, T, num_ctas, pl);
    if (s) return s;
    if (c->B > 0 && !n_new) return fail(KVC_ERR_ARG, "n_new is null");
    for (int b = 0; b < c->B; ++b) {
        if (n_new[b] < 0 || n_new[b] > T)
            return fail(KVC_ERR_SHAPE, "row %d: n_new = %d outside 0..%d", b, n_new[b], T);
        if (n_new[b] > lens_after[b])
            return fail(KVC_ERR_SHAPE, "row %d: n_new = %d exceeds the row length %lld", b, n_new[b],
                        static_cast<long long>(lens_after[b]));
    }
    if (c->B > 0 && T > 0) {
        if (!q || !out) return fail(KVC_ERR_ARG, "q / out is null");
        if (!aligned16(q) || !aligned16(out)) return fail(KVC_ERR_ARG, "q / out not 16-byte aligned");
    }
    return ok();
}

// ---------------------------------------------------------------------------
// Launches (arguments already validated)
// ---------------------------------------------------------------------------

// The layer's FP8 scales into a split-KV parameter block (no-op for bf16).
void set_decode_scales(const kvc_cache* c, int layer, DecodeParams* p) {
    if (c->dtype != KVC_FP8_E4M3) return;
    for (int h = 0; h < c->Hkv; ++h) {
        p->kscale[h] = c->kscale[static_cast<size_t>(layer) * c->Hkv + h];
        p->vscale[h] = c->vscale[static_cast<size_t>(layer) * c->Hkv + h];
    }
}

kvc_status do_append(kvc_cache* c, int layer, const void* k_new, const void* v_new, int T, const int32_t* n_new,
                     int max_n, cudaStream_t stream) {
    if (max_n == 0) return ok();
    static_assert(sizeof(AppendParams) < 32000, "kernel parameter block too large");
    AppendParams p;
    p.k_new = static_cast<const uint8_t*>(k_new);
    p.v_new = static_cast<const uint8_t*>(v_new);
    p.k_cache = static_cast<uint8_t*>(c->k[layer]);
    p.v_cache = static_cast<uint8_t*>(c->v[layer]);
    p.B = c->B;
    p.Hkv = c->Hkv;
    p.T = T;
    p.max_len = c->max_len;
    p.fp8 = c->dtype == KVC_FP8_E4M3 ? 1 : 0;
    p.row_bytes = c->d * (p.fp8 ? 2 : c->esize);  // source rows (bf16 for an FP8 cache)
    p.ring = c->ring ? 1 : 0;
    p.pg = c->pg;
    if (p.fp8)
        for (int h = 0; h < c->Hkv; ++h) {
            p.kscale[h] = c->kscale[static_cast<size_t>(layer) * c->Hkv + h];
            p.vscale[h] = c->vscale[static_cast<size_t>(layer) * c->Hkv + h];
        }
    const int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    for (int b = 0; b < c->B; ++b) {
        p.lens[b] = static_cast<int>(lens[b]);
        p.n_new[b] = n_new[b];
    }
    cudaError_t e = launch_append(p, max_n, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    ++c->launches;
    return ok();
}

// With k_new / v_new given (bf16, warps owning whole tiles) the attention
// kernel also performs the append; *main_enqueued tells whether the attention
// kernel was enqueued (so a caller can undo its length update if not).
kvc_status do_attention(kvc_cache* c, int layer, const void* q, const AttnPlan& pl, const int32_t* n_new, void* out,
                        void* ws, size_t ws_bytes, cudaStream_t stream, const void* k_new = nullptr,
                        const void* v_new = nullptr, bool* main_enqueued = nullptr, const uint64_t* anc = nullptr) {
    if (main_enqueued) *main_enqueued = false;
    const int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    if (c->B == 0 || pl.T == 0) return ok();
    if (pl.generic) {
        static_assert(sizeof(F32Params) < 32000, "kernel parameter block too large");
        F32Params p;
        p.q = q;
        p.k_cache = c->k[layer];
        p.v_cache = c->v[layer];
        p.out = out;
        p.kind = c->dtype == KVC_FP8_E4M3 ? 2 : (c->dtype == KVC_BF16 ? 1 : 0);
        for (int h = 0; h < c->Hkv && p.kind == 2; ++h) {
            p.kscale[h] = c->kscale[static_cast<size_t>(layer) * c->Hkv + h];
            p.vscale[h] = c->vscale[static_cast<size_t>(layer) * c->Hkv + h];
        }
        p.B = c->B;
        p.Hq = pl.Hq;
        p.Hkv = c->Hkv;
        p.G = pl.G;
        p.T = pl.T;
        p.max_len = c->max_len;
        p.d = c->d;
        p.R = pl.R;
        p.window = c->window;
        p.ring = c->ring ? 1 : 0;
        p.tree = anc ? 1 : 0;
        if (anc) std::copy(anc, anc + static_cast<size_t>(c->B) * pl.T, p.anc);
        p.pg = c->pg;
        p.scale = 1.0f / sqrtf(static_cast<float>(c->d));
        p.splits = pl.splits;
        p.partials = nullptr;
        p.counters = nullptr;
        if (pl.splits > 1) {
            p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.ws_err);
            p.counters = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + kWsCounterOffset);
            if (ws != c->last_ws) {  // the counters start at zero and return to it after each call
                cudaError_t e = cudaMemsetAsync(ws, 0, pl.ws_err, stream);
                if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
                c->last_ws = ws;
            }
        }
        for (int b = 0; b < c->B; ++b) {
            p.prior[b] = static_cast<int>(lens[b] - n_new[b]);
            p.n_new[b] = n_new[b];
        }
        cudaError_t e = launch_attn_f32(p, stream);
        if (e != cudaSuccess) return cuda_fail(e, "generic attention launch");
        ++c->launches;
        return ok();
    }

    kvc_status s = encode_layer_maps(c, layer);
    if (s) return s;
    if (pl.R > tc_min_rows(c) && k_new == nullptr && anc == nullptr && c->max_len <= kTcMaxLen && tc_capable(c)) {
        // Many query rows per KV head: tensor-core kernel, one CTA per piece.
        // Work items are (b, kvh, row block, pair of 128-row tiles): with
        // T >= 128, 128 positions of two query heads (mode 0); with T < 128 the
        // G*T rows r = g*T + t of the KV head packed into 128-row tiles (mode 1),
        // or all in one tile whose two TMEM buffers take alternate key tiles
        // (mode 2, G*T <= 128).  An item's key tiles cost its tile count each
        // (one in mode 2), plus a fixed start-up cost per CTA.  The launch order
        // comes from a longest-first list schedule simulated on the SMs (the
        // block scheduler hands the next CTA to the first SM that frees up):
        // an item that would run past the SMs' common finishing time is cut
        // there, and the rest of it is scheduled like any other item.  The
        // pieces of a cut item leave partials that its last piece merges.
        // Items of equal length (the 128-position blocks and head pairs that
        // read the same K/V) stay side by side, so their K/V tiles are read
        // from HBM about once and then hit in L2.
        static_assert(sizeof(PrefillParams) < 32000, "kernel parameter block too large");
        struct WorkItem {
            int code, kt0, nkt, nh;  // key tiles kt0 .. nkt - 1 (absolute position / 128)
        };
        std::vector<WorkItem> items;
        PrefillParams pp;
        pp.q = q;
        pp.out = out;
        pp.err = static_cast<int*>(ws);
        pp.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.ws_err + pl.ws_plan);
        pp.B = c->B;
        pp.Hq = pl.Hq;
        pp.Hkv = c->Hkv;
        pp.G = pl.G;
        pp.T = pl.T;
        pp.max_len = c->max_len;
        pp.mode = pl.T >= 128 ? 0 : (pl.R <= 128 ? 2 : 1);
        pp.fp8 = c->dtype == KVC_FP8_E4M3 ? 1 : 0;
        if (pp.fp8)
            for (int h = 0; h < c->Hkv; ++h) {
                pp.kscale[h] = c->kscale[static_cast<size_t>(layer) * c->Hkv + h];
                pp.vscale[h] = c->vscale[static_cast<size_t>(layer) * c->Hkv + h];
            }
        pp.ntb = pp.mode == 0 ? (pl.T + 127) / 128 : 1;
        pp.npair = pp.mode == 0 ? (pl.G + 1) / 2 : (pl.R + 255) / 256;
        pp.window = c->window;
        pp.ring = c->ring ? 1 : 0;
        pp.pg = c->pg;
        pp.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(c->d)));
        for (int b = 0; b < c->B; ++b) {
            pp.prior[b] = static_cast<int>(lens[b] - n_new[b]);
            pp.n_new[b] = n_new[b];
            for (int kvh = 0; kvh < c->Hkv && pp.mode != 0 && n_new[b] > 0; ++kvh) {
                // Packed rows: the last key any row sees is prior + min(T, n_new) - 1,
                // and the first key any row's window starts at is prior - W + 1 or later.
                const int kmax = pp.prior[b] + std::min(pl.T, static_cast<int>(n_new[b])) - 1;
                const int kfirst = c->window > 0 ? std::max(0, pp.prior[b] - c->window + 1) : 0;
                for (int pr = 0; pr < pp.npair; ++pr) {
                    const int code = (b * c->Hkv + kvh) * pp.npair + pr;
                    const int cost = pp.mode == 2 ? 1 : std::min(2, (pl.R - pr * 256 + 127) / 128);
                    items.push_back({code, kfirst / 128, kmax / 128 + 1, cost});
                }
            }
            for (int kvh = 0; kvh < c->Hkv && pp.mode == 0; ++kvh)
                for (int tb = 0; tb < pp.ntb; ++tb) {
                    const int t0 = tb * 128;
                    if (t0 >= n_new[b]) continue;
                    const int kmax = pp.prior[b] + std::min(t0 + 127, static_cast<int>(n_new[b]) - 1);
                    // First key any query of the block sees: its first query's window start.
                    const int kfirst = c->window > 0 ? std::max(0, pp.prior[b] + t0 - c->window + 1) : 0;
                    for (int pr = 0; pr < pp.npair; ++pr) {
                        const int code = ((b * c->Hkv + kvh) * pp.ntb + tb) * pp.npair + pr;
                        items.push_back({code, kfirst / 128, kmax / 128 + 1, std::min(2, pl.G - 2 * pr)});
                    }
                }
        }
        const size_t slot_bytes = static_cast<size_t>(2) * 128 * (kHeadDimBf16 + 4) * sizeof(float);
        const long long slot_room =
            std::min<long long>(kMaxPrefillSlots, static_cast<long long>((ws_bytes - pl.ws_err - pl.ws_plan) / slot_bytes));
        const int nsm = std::max(1, c->num_sms);
        // Items per launch, leaving room for the pieces that cuts add.
        const size_t chunk = static_cast<size_t>(kMaxPrefillPieces - std::min(nsm, kMaxPrefillPieces / 4));
        bool launched = false;
        if (!items.empty()) {
            CUtensorMap tmQ;
            if ((s = encode_rows_map(&tmQ, q, static_cast<cuuint64_t>(c->B) * pl.Hq * pl.T, 128))) return s;
            if (ws != c->last_ws) {
                cudaError_t e = cudaMemsetAsync(ws, 0, pl.ws_err, stream);
                if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
                c->last_ws = ws;
            }
            for (size_t i0 = 0; i0 < items.size(); i0 += chunk) {
                const size_t i1 = std::min(items.size(), i0 + chunk);
                const int n_items = static_cast<int>(i1 - i0);
                // Per-CTA start-up cost in (tile x head) units and the shortest piece a cut
                // may leave.  A per-CTA timeline of the chunked-prefill shape fits a piece's
                // time as 5.1 us + 1.02 us per tile x head, so start-up is 5 units (13 and 8
                // were 1 to 10 % slower); pieces of 16 tiles were 1 to 4 % slower, pieces of
                // 4 tiles the same.
                constexpr long long kStartCost = 5;
                constexpr int kMinPieceTiles = 8;
                long long W = 0;
                for (size_t k = i0; k < i1; ++k)
                    W += static_cast<long long>(items[k].nkt - items[k].kt0) * items[k].nh + kStartCost;
                const long long target = W / nsm + kStartCost;  // the SMs' common finishing time
                // Remaining parts of items, longest first (ties: item order).
                struct Part {
                    long long cost;
                    int item, lo;
                    bool operator<(const Part& o) const { return cost != o.cost ? cost < o.cost : item > o.item; }
                };
                std::priority_queue<Part> parts;
                for (int k = 0; k < n_items; ++k) {
                    const WorkItem& it = items[i0 + k];
                    parts.push({static_cast<long long>(it.nkt - it.kt0) * it.nh, k, it.kt0});
                }
                using Sm = std::pair<long long, int>;  // (busy until, SM)
                std::priority_queue<Sm, std::vector<Sm>, std::greater<Sm>> sms;
                for (int m = 0; m < nsm; ++m) sms.push({0, m});
                struct Placed {
                    long long start;
                    int seq, item, lo, hi;
                };
                std::vector<Placed> placed;
                int cuts = 0;
                while (!parts.empty()) {
                    const Part pt = parts.top();
                    parts.pop();
                    const WorkItem& it = items[i0 + pt.item];
                    const Sm sm = sms.top();
                    sms.pop();
                    int hi = it.nkt;
                    const long long room = target - sm.first - kStartCost;  // work that fits before the target
                    const int fit = static_cast<int>(std::max(0ll, room) / it.nh);
                    const bool can_cut = n_items + cuts + 1 <= kMaxPrefillPieces && 2ll * (cuts + 1) <= slot_room;
                    if (pt.cost + kStartCost > target - sm.first && can_cut && fit >= kMinPieceTiles &&
                        it.nkt - (pt.lo + fit) >= kMinPieceTiles) {
                        hi = pt.lo + fit;
                        ++cuts;
                        parts.push({static_cast<long long>(it.nkt - hi) * it.nh, pt.item, hi});
                    }
                    placed.push_back({sm.first, static_cast<int>(placed.size()), pt.item, pt.lo, hi});
                    sms.push({sm.first + kStartCost + static_cast<long long>(hi - pt.lo) * it.nh, sm.second});
                }
                std::sort(placed.begin(), placed.end(), [](const Placed& x, const Placed& y) {
                    return x.start != y.start ? x.start < y.start : x.seq < y.seq;
                });
                // Slots: the pieces of a cut item take consecutive slots.
                std::vector<int> npieces(n_items, 0), slot0(n_items, -1), seen(n_items, 0);
                for (const Placed& pc : placed) ++npieces[pc.item];
                int slots = 0;
                for (int k = 0; k < n_items; ++k)
                    if (npieces[k] > 1) {
                        slot0[k] = slots;
                        slots += npieces[k];
                    }
                pp.n_pieces = static_cast<int>(placed.size());
                for (int q2 = 0; q2 < pp.n_pieces; ++q2) {
                    const Placed& pc = placed[q2];
                    const WorkItem& it = items[i0 + pc.item];
                    pp.piece_code[q2] = static_cast<uint32_t>(it.code);
                    pp.piece_tiles[q2] = static_cast<uint32_t>(pc.lo) | (static_cast<uint32_t>(pc.hi) << 16);
                    if (npieces[pc.item] > 1) {
                        const int kidx = seen[pc.item]++;
                        pp.piece_aux[q2] = static_cast<uint32_t>(slot0[pc.item] + kidx) |
                                           (static_cast<uint32_t>(kidx) << 12) |
                                           (static_cast<uint32_t>(npieces[pc.item]) << 22);
                    } else {
                        pp.piece_aux[q2] = static_cast<uint32_t>(kPrefillNoSlot);
                    }
                }
                cudaError_t e = launch_prefill_tc(pp, tmQ, c->tmK128[layer], c->tmV128[layer], stream);
                if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
                ++c->launches;
                launched = true;
                if (main_enqueued) *main_enqueued = true;
            }
        }
        if (launched) return ok();
        // otherwise (no rows to attend, or no room for the partials): the split-KV path below
    }

    // bf16 split-KV path
    static_assert(sizeof(DecodeParams) < 32000, "kernel parameter block too large");
    DecodeParams p;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    p.err = reinterpret_cast<int*>(wsb);
    p.partials = reinterpret_cast<float*>(wsb + pl.ws_err + pl.ws_plan);
    p.dplan = nullptr;
    p.q = q;
    p.out = out;
    p.B = c->B;
    p.Hq = pl.Hq;
    p.Hkv = c->Hkv;
    p.G = pl.G;
    p.T = pl.T;
    p.max_len = c->max_len;
    p.R = pl.R;
    p.RPB = pl.RPB;
    p.RB = pl.RB;
    p.NB = pl.NB;
    p.part_rows = pl.part_rows;
    p.append_new = (k_new != nullptr && v_new != nullptr) ? 1 : 0;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = c->k[layer];
    p.v_cache = c->v[layer];
    p.Tn = pl.T;
    p.window = c->window;
    p.ring = c->ring ? 1 : 0;
    p.pg = c->pg;
    set_decode_scales(c, layer, &p);
    p.anc = nullptr;
    if (anc) {
        // The masks go to the workspace (the parameter block stays small).
        uint64_t* dev_anc = reinterpret_cast<uint64_t*>(wsb + pl.ws_err + round_up(sizeof(DevicePlan), 256));
        cudaError_t e = cudaMemcpyAsync(dev_anc, anc, static_cast<size_t>(c->B) * pl.T * sizeof(uint64_t),
                                        cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "copying the draft-tree masks");
        p.anc = dev_anc;
    }
    p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(c->d)));
    long long tiles = 0;
    for (int b = 0; b < c->B; ++b) {
        p.prior[b] = static_cast<int>(lens[b] - n_new[b]);
        p.n_new[b] = n_new[b];
    }
    for (int b = 0; b < c->B; ++b) {
        for (int rb = 0; rb < pl.RB; ++rb) {
            // Extent of the row block: one past the largest visible key of its
            // valid rows; with a window its keys start at the window of its
            // earliest query (tiles before that are never scheduled).
            int extent = 0, qmin = 0x7fffffff;
            const int r0 = rb * pl.RPB, r1 = std::min(pl.R, r0 + pl.RPB);
            if (r1 - r0 >= pl.T) {
                if (n_new[b] > 0) {
                    extent = p.prior[b] + std::min(pl.T, static_cast<int>(n_new[b]));
                    qmin = p.prior[b];
                }
            } else {
                for (int r = r0; r < r1; ++r) {
                    const int t = r % pl.T;
                    if (t < n_new[b]) {
                        extent = std::max(extent, p.prior[b] + t + 1);
                        qmin = std::min(qmin, p.prior[b] + t);
                    }
                }
            }
            const int kfirst = (extent > 0 && c->window > 0) ? std::max(0, qmin - c->window + 1) : 0;
            const int kt = key_tile_keys(c->d, c->dtype == KVC_FP8_E4M3);
            const int first_tile = kfirst / kt;
            const int ntiles = extent > 0 ? (extent - 1) / kt + 1 - first_tile : 0;
            p.gstart[b * pl.RB + rb] = static_cast<int>(tiles);
            tiles += static_cast<long long>(ntiles) * c->Hkv;
        }
    }
    if (tiles > 0x7fffffffll) return fail(KVC_ERR_ARG, "too many key tiles in one call");
    p.gstart[pl.NB] = static_cast<int>(tiles);
    p.total_tiles = static_cast<int>(tiles);
    // At most one CTA per SM, and never more CTAs than tiles: then every CTA
    // owns at least one tile, so the CTAs covering a unit's tiles are exactly
    // the contiguous range cta_of(first tile) .. cta_of(last tile), all of
    // which contribute a partial.
    const int grid = static_cast<int>(std::max(1ll, std::min<long long>(c->num_sms, tiles)));
    p.num_ctas = grid;

    // Does any unit need the combine kernel?  A unit is written in full by the
    // attention kernel when all its tiles fall in one CTA (CTA i owns tiles
    // floor(iN/P) .. floor((i+1)N/P)-1, so tile x belongs to CTA
    // ((x+1)P - 1) / N) and, when warps own whole tiles, it is one tile.
    bool need_combine = false;
    {
        const long long N = tiles, P = grid;
        for (int q = 0; q < pl.NB && !need_combine; ++q) {
            const int nt = (p.gstart[q + 1] - p.gstart[q]) / c->Hkv;
            if (nt == 0) continue;
            if (pl.ways > 1 && nt > 1) {
                need_combine = true;
                break;
            }
            for (int kvh = 0; kvh < c->Hkv; ++kvh) {
                const long long us = p.gstart[q] + static_cast<long long>(kvh) * nt, ue = us + nt - 1;
                if (((us + 1) * P - 1) / N != ((ue + 1) * P - 1) / N) {
                    need_combine = true;
                    break;
                }
            }
        }
    }

    if (ws != c->last_ws) {
        // New workspace: clear the error word once; kernels only ever set it.
        cudaError_t e = cudaMemsetAsync(ws, 0, pl.ws_err, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
        c->last_ws = ws;
    }
    cudaError_t e =
        launch_decode_bf16(p, c->tmK[layer], c->tmV[layer], pl.mt, grid, c->dtype == KVC_FP8_E4M3, c->d, stream);
    if (e != cudaSuccess) return cuda_fail(e, "split-KV attention launch");
    ++c->launches;
    if (main_enqueued) *main_enqueued = true;
    if (need_combine) {
        static_assert(sizeof(CombineParams) < 32000, "kernel parameter block too large");
        CombineParams cp;
        cp.dplan = nullptr;
        cp.partials = p.partials;
        cp.out = out;
        cp.d = c->d;
        cp.Hq = pl.Hq;
        cp.Hkv = c->Hkv;
        cp.G = pl.G;
        cp.T = pl.T;
        cp.R = pl.R;
        cp.RPB = pl.RPB;
        cp.RB = pl.RB;
        cp.NB = pl.NB;
        cp.ways = pl.ways;
        cp.part_rows = pl.part_rows;
        cp.total_tiles = p.total_tiles;
        cp.num_ctas = grid;
        for (int b = 0; b < c->B; ++b) cp.n_new[b] = n_new[b];
        for (int q = 0; q <= pl.NB; ++q) cp.gstart[q] = p.gstart[q];
        for (int i = 0; i <= grid; ++i) cp.cta_start[i] = static_cast<int>(static_cast<long long>(i) * tiles / grid);
        e = launch_combine_bf16(cp, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split-KV combine launch");
        ++c->launches;
    }
    (void)ws_bytes;
    return ok();
}

kvc_status check_workspace(const kvc_cache* c, const AttnPlan& pl, const void* ws, size_t ws_bytes) {
    if (c->B == 0 || pl.T == 0 || pl.ws_total == 0) return ok();  // (the generic kernel may need none)
    if (!ws) return fail(KVC_ERR_WORKSPACE, "workspace is null (need %zu bytes)", pl.ws_total);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(KVC_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (ws_bytes < pl.ws_total)
        return fail(KVC_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, pl.ws_total);
    return ok();
}

// Copy a workspace's error word to *code after the stream's work, clear it
// when set, and map the code to a status.
kvc_status read_error_word(void* word, cudaStream_t st, int32_t* code) {
    *code = 0;
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    *code = v;
    if (v != 0) {
        e = cudaMemsetAsync(word, 0, sizeof v, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        if (v == kDevOverflow)
            return fail(KVC_ERR_OVERFLOW, "a device-resident step was rejected: a row would pass max_len or n_new "
                                          "was outside 0..T (nothing was written, lengths unchanged)");
        if (v == kDevBadPage)
            return fail(KVC_ERR_ARG, "a block-table entry under an attended or appended position was outside "
                                     "0..num_pages-1 (not dereferenced; the call's output is not valid)");
        return fail(KVC_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait expired (code %d)", v);
    }
    return ok();
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================



// Ancestor masks of a draft tree ("Write the causal mask for a decode
// step...", "What interviewers probe next": tree-based speculative decoding):
// query t of row b may see chunk token u iff u is on t's path to the root.
// parents[b * T + t] in -1 .. t - 1 for t < n_new[b] (a parent precedes its
// child; -1: the token hangs directly off the cached prefix).
kvc_status tree_masks(const kvc_cache* c, const AttnPlan& pl, const int32_t* n_new, const int32_t* parents,
                      std::vector<uint64_t>* anc) {
    if (!parents && c->B > 0) return fail(KVC_ERR_ARG, "parents is null");
    if (pl.T > 64) return fail(KVC_ERR_SHAPE, "a draft tree takes at most 64 tokens per row (T = %d)", pl.T);
    if (static_cast<long long>(c->B) * pl.T > kMaxTreeQueries)
        return fail(KVC_ERR_SHAPE, "B * T = %lld draft tokens exceed %d", static_cast<long long>(c->B) * pl.T,
                    kMaxTreeQueries);
    if (c->window > 0 || c->ring) return fail(KVC_ERR_ARG, "a draft tree does not combine with a window");
    if (tc_capable(c) && pl.R > 64)
        return fail(KVC_ERR_SHAPE, "a bf16 / fp8 draft tree takes G * T <= 64 query rows per KV head (G * T = %d)", pl.R);
    anc->assign(static_cast<size_t>(c->B) * pl.T, 0);
    for (int b = 0; b < c->B; ++b)
        for (int t = 0; t < n_new[b]; ++t) {
            const int pa = parents[static_cast<size_t>(b) * pl.T + t];
            if (pa < -1 || pa >= t)
                return fail(KVC_ERR_SHAPE, "row %d: parent %d of draft token %d outside -1..%d", b, pa, t, t - 1);
            (*anc)[static_cast<size_t>(b) * pl.T + t] =
                (1ull << t) | (pa >= 0 ? (*anc)[static_cast<size_t>(b) * pl.T + pa] : 0ull);
        }
    return ok();
}

// Calls that read or write the host copy of the lengths refuse while the
// device copy is authoritative.
kvc_status check_host_lens(const kvc_cache* c) {
    if (c && c->lens_on_device)
        return fail(KVC_ERR_ARG, "the lengths live on the device (kvc_lens_to_device); call kvc_lens_from_device first");
    return ok();
}

// Helpers of the host-buffer calls (kvc_append_attention_host).
namespace {

// Bytes of one element of q, k_new, v_new and out (bf16 for an FP8 cache).
size_t io_esize(const kvc_cache* c) { return c->dtype == KVC_FP8_E4M3 ? 2 : static_cast<size_t>(c->esize); }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Streams, events and two staging slots of at least `bytes` each.  A slot that
// grows is freed only after the calls that used it have finished with it.
kvc_status ensure_host_staging(kvc_cache* c, size_t bytes) {
    cudaError_t e = cudaSuccess;
    if (!c->h2d) {
        cudaStream_t h2d = nullptr, d2h = nullptr;
        e = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking);
        for (auto& hs : c->hslot)
            for (cudaEvent_t* ev : {&hs.in_ready, &hs.computed, &hs.out_done})
                if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            // Leave nothing half made: the next call starts over.
            for (auto& hs : c->hslot)
                for (cudaEvent_t* ev : {&hs.in_ready, &hs.computed, &hs.out_done})
                    if (*ev) {
                        cudaEventDestroy(*ev);
                        *ev = nullptr;
                    }
            if (h2d) cudaStreamDestroy(h2d);
            if (d2h) cudaStreamDestroy(d2h);
            return cuda_fail(e, "host-call streams / events");
        }
        c->h2d = h2d;
        c->d2h = d2h;
    }
    for (auto& hs : c->hslot) {
        if (hs.bytes >= bytes) continue;
        if (hs.buf) {
            e = cudaEventSynchronize(hs.computed);
            if (e == cudaSuccess) e = cudaEventSynchronize(hs.out_done);
            if (e == cudaSuccess) e = cudaStreamSynchronize(c->h2d);
            if (e == cudaSuccess) e = cudaFree(hs.buf);
            hs.buf = nullptr;
            hs.bytes = 0;
            if (e != cudaSuccess) return cuda_fail(e, "host-call staging release");
        }
        e = cudaMalloc(&hs.buf, bytes);
        if (e != cudaSuccess) {
            hs.buf = nullptr;
            return cuda_fail(e, "host-call staging allocation");
        }
        hs.bytes = bytes;
    }
    return ok();
}

// Copy positions t < n_new[b] of a [B, H, T, d] tensor: the whole tensor in
// one copy when every row is full, else one 2-D copy per row (H runs of
// n_new[b] rows of `row_bytes`, pitch T rows).  Nothing else is touched.
cudaError_t copy_chunk(void* dst, const void* src, int B, int H, int T, size_t row_bytes, const int32_t* n_new,
                       cudaMemcpyKind kind, cudaStream_t st) {
    bool full = true;
    for (int b = 0; b < B; ++b) full = full && n_new[b] == T;
    const size_t pitch = static_cast<size_t>(T) * row_bytes, per_row = static_cast<size_t>(H) * pitch;
    if (full) return cudaMemcpyAsync(dst, src, static_cast<size_t>(B) * per_row, kind, st);
    for (int b = 0; b < B; ++b) {
        if (n_new[b] == 0) continue;
        cudaError_t e = cudaMemcpy2DAsync(static_cast<char*>(dst) + b * per_row, pitch,
                                          static_cast<const char*>(src) + b * per_row, pitch,
                                          static_cast<size_t>(n_new[b]) * row_bytes, H, kind, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

extern "C" {

kvc_status kvc_create(kvc_cache** out, int layers, int batch, int kv_heads, int max_len, int head_dim,
                      kvc_dtype dtype, void* const* k_bufs, void* const* v_bufs) {
    if (!out) return fail(KVC_ERR_ARG, "out is null");
    *out = nullptr;
    if (layers < 1 || batch < 0 || kv_heads < 1 || max_len < 1 || head_dim < 1)
        return fail(KVC_ERR_ARG, "bad geometry: layers=%d batch=%d kv_heads=%d max_len=%d head_dim=%d", layers, batch,
                    kv_heads, max_len, head_dim);
    if (batch > KVC_MAX_BATCH) return fail(KVC_ERR_ARG, "batch %d > %d", batch, KVC_MAX_BATCH);
    if (dtype != KVC_F32 && dtype != KVC_BF16 && dtype != KVC_FP8_E4M3)
        return fail(KVC_ERR_ARG, "unknown dtype %d", static_cast<int>(dtype));
    const int esize = dtype == KVC_F32 ? 4 : (dtype == KVC_BF16 ? 2 : 1);
    if ((head_dim * esize) % 16 != 0) return fail(KVC_ERR_ARG, "head_dim * element size must be a multiple of 16");
    if (head_dim > 256) return fail(KVC_ERR_ARG, "head_dim %d > 256", head_dim);
    if (dtype == KVC_FP8_E4M3 && kv_heads > kMaxScaleHeads)
        return fail(KVC_ERR_ARG, "fp8 caches take at most %d KV heads", kMaxScaleHeads);
    const long long rows = static_cast<long long>(batch) * kv_heads * max_len;
    if (rows + 2 * kKeyTile >= (1ll << 31)) return fail(KVC_ERR_ARG, "batch * kv_heads * max_len too large");
    if (!k_bufs || !v_bufs) return fail(KVC_ERR_ARG, "k_bufs / v_bufs is null");
    for (int l = 0; l < layers; ++l) {
        if (!k_bufs[l] || !v_bufs[l]) return fail(KVC_ERR_ARG, "layer %d buffer is null", l);
        if (!aligned16(k_bufs[l]) || !aligned16(v_bufs[l]))
            return fail(KVC_ERR_ARG, "layer %d buffer not 16-byte aligned", l);
    }
    kvc_cache* c = new kvc_cache;
    c->layers = layers;
    c->B = batch;
    c->Hkv = kv_heads;
    c->max_len = max_len;
    c->d = head_dim;
    c->dtype = dtype;
    c->esize = esize;
    c->k.assign(k_bufs, k_bufs + layers);
    c->v.assign(v_bufs, v_bufs + layers);
    c->lens.assign(static_cast<size_t>(layers) * batch, 0);
    c->tmK.resize(layers);
    c->tmV.resize(layers);
    c->tmK128.resize(layers);
    c->tmV128.resize(layers);
    c->tm_ready.assign(layers, 0);
    c->kscale.assign(static_cast<size_t>(layers) * kv_heads, 1.0f);
    c->vscale.assign(static_cast<size_t>(layers) * kv_heads, 1.0f);
    *out = c;
    return ok();
}

kvc_status kvc_set_kv_scales(kvc_cache* c, int layer, const float* k_scale, const float* v_scale) {
    if (!c) return fail(KVC_ERR_ARG, "null handle");
    if (c->dtype != KVC_FP8_E4M3) return fail(KVC_ERR_ARG, "scales apply to fp8 caches only");
    if (layer < 0 || layer >= c->layers) return fail(KVC_ERR_ARG, "layer %d out of range", layer);
    if (!k_scale || !v_scale) return fail(KVC_ERR_ARG, "k_scale / v_scale is null");
    for (int h = 0; h < c->Hkv; ++h)
        if (!(std::isfinite(k_scale[h]) && std::isfinite(v_scale[h]) && k_scale[h] > 0.f && v_scale[h] > 0.f))
            return fail(KVC_ERR_ARG, "head %d: scales must be positive and finite", h);
    if (c->lens_on_device) return fail(KVC_ERR_ARG, "lengths are on the device; call kvc_lens_from_device first");
    for (int b = 0; b < c->B; ++b)
        if (c->lens[static_cast<size_t>(layer) * c->B + b] != 0)
            return fail(KVC_ERR_ARG, "layer %d holds data: scales change only while it is empty", layer);
    std::copy(k_scale, k_scale + c->Hkv, c->kscale.begin() + static_cast<size_t>(layer) * c->Hkv);
    std::copy(v_scale, v_scale + c->Hkv, c->vscale.begin() + static_cast<size_t>(layer) * c->Hkv);
    return ok();
}

kvc_status kvc_create_paged(kvc_cache** out, int layers, int batch, int kv_heads, int page_size, int num_pages,
                            int max_pages_per_row, int head_dim, kvc_dtype dtype, void* const* k_bufs,
                            void* const* v_bufs, const int32_t* block_table) {
    if (!out) return fail(KVC_ERR_ARG, "out is null");
    *out = nullptr;
    if (page_size < 1 || num_pages < 1 || max_pages_per_row < 1)
        return fail(KVC_ERR_ARG, "bad paging: page_size=%d num_pages=%d max_pages_per_row=%d", page_size, num_pages,
                    max_pages_per_row);
    if (dtype != KVC_F32 && head_dim == kHeadDimBf16 && page_size % 128 != 0)
        return fail(KVC_ERR_ARG, "bf16 and fp8 pages of head_dim %d hold a multiple of 128 tokens (key tiles never cross a page)",
                    kHeadDimBf16);
    if (dtype == KVC_BF16 && head_dim == kHeadDimSmall && page_size % key_tile_keys(kHeadDimSmall, false) != 0)
        return fail(KVC_ERR_ARG, "bf16 pages of head_dim %d hold a multiple of %d tokens (key tiles never cross a page)",
                    kHeadDimSmall, key_tile_keys(kHeadDimSmall, false));
    if (batch > 0 && !block_table) return fail(KVC_ERR_ARG, "block_table is null");
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0) return fail(KVC_ERR_ARG, "block_table not 4-byte aligned");
    const long long cap = static_cast<long long>(max_pages_per_row) * page_size;
    if (cap >= (1ll << 30)) return fail(KVC_ERR_ARG, "max_pages_per_row * page_size too large");
    if (static_cast<long long>(num_pages) * kv_heads * page_size + 2 * kKeyTile >= (1ll << 31))
        return fail(KVC_ERR_ARG, "num_pages * kv_heads * page_size too large");
    if (static_cast<long long>(batch) * max_pages_per_row >= (1ll << 31))
        return fail(KVC_ERR_ARG, "batch * max_pages_per_row too large");
    // The ordinary handle over the logical geometry; the buffers are pages.
    kvc_status s = kvc_create(out, layers, batch, kv_heads, static_cast<int>(cap), head_dim, dtype, k_bufs, v_bufs);
    if (s) return s;
    (*out)->pg = Paging{block_table, page_size, max_pages_per_row, num_pages};
    return ok();
}

void kvc_destroy(kvc_cache* c) {
    if (c && c->h2d) {
        // Host-buffer calls may still be copying: let them finish first.
        cudaStreamSynchronize(c->h2d);
        cudaStreamSynchronize(c->d2h);
        for (auto& hs : c->hslot) {
            if (hs.computed) cudaEventSynchronize(hs.computed);
            if (hs.buf) cudaFree(hs.buf);
            for (cudaEvent_t e : {hs.in_ready, hs.computed, hs.out_done})
                if (e) cudaEventDestroy(e);
        }
        cudaStreamDestroy(c->h2d);
        cudaStreamDestroy(c->d2h);
    }
    delete c;
}

kvc_status kvc_append(kvc_cache* c, int layer, const void* k_new, const void* v_new, int T, const int32_t* n_new,
                      void* stream) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    int max_n = 0;
    kvc_status s = validate_append(c, layer, k_new, v_new, T, n_new, &max_n);
    if (s) return s;
    if (max_n > 0) {
        s = ensure_device(c);
        if (s) return s;
        s = do_append(c, layer, k_new, v_new, T, n_new, max_n, static_cast<cudaStream_t>(stream));
        if (s) return s;
    }
    int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    for (int b = 0; b < c->B; ++b) lens[b] += n_new[b];
    return ok();
}

size_t kvc_workspace_bytes(const kvc_cache* c, int q_heads, int T) {
    if (!c) return 0;
    kvc_cache* mc = const_cast<kvc_cache*>(c);
    if (ensure_device(mc) != KVC_OK) return 0;
    AttnPlan pl;
    if (plan_shape(c, q_heads, T, c->num_sms, &pl) != KVC_OK) return 0;
    return pl.ws_total;
}

static kvc_status gqa_attention_impl(kvc_cache* c, int layer, const void* q, int q_heads, int T, const int32_t* n_new,
                              const int32_t* parents, void* out, void* workspace, size_t workspace_bytes,
                              void* stream) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    kvc_status s = check_layer(c, layer);
    if (s) return s;
    AttnPlan pl;
    const int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    s = validate_attention(c, layer, q, q_heads, T, n_new, out, lens, &pl, 0);
    if (s) return s;
    std::vector<uint64_t> anc;  // (validated before any CUDA call)
    if (parents) {
        s = tree_masks(c, pl, n_new, parents, &anc);
        if (s) return s;
    }
    if (c->B > 0 && T > 0) {
        s = ensure_device(c);
        if (s) return s;
        s = plan_shape(c, q_heads, T, c->num_sms, &pl);
        if (s) return s;
    }
    s = check_workspace(c, pl, workspace, workspace_bytes);
    if (s) return s;
    if (c->B == 0 || T == 0) return ok();
    s = ensure_device(c);
    if (s) return s;
    return do_attention(c, layer, q, pl, n_new, out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                        nullptr, nullptr, nullptr, parents ? anc.data() : nullptr);
}

static kvc_status append_attention_impl(kvc_cache* c, int layer, const void* q, const void* k_new, const void* v_new,
                                 int q_heads, int T, const int32_t* n_new, const int32_t* parents, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    int max_n = 0;
    kvc_status s = validate_append(c, layer, k_new, v_new, T, n_new, &max_n);
    if (s) return s;
    // Validate the attention step against the lengths the append will produce.
    std::vector<int64_t> after(c->B);
    const int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    for (int b = 0; b < c->B; ++b) after[b] = lens[b] + n_new[b];
    AttnPlan pl;
    s = validate_attention(c, layer, q, q_heads, T, n_new, out, after.data(), &pl, 0);
    if (s) return s;
    std::vector<uint64_t> anc;  // (validated before any CUDA call)
    if (parents) {
        s = tree_masks(c, pl, n_new, parents, &anc);
        if (s) return s;
    }
    if (c->B > 0 && T > 0) {
        s = ensure_device(c);
        if (s) return s;
        s = plan_shape(c, q_heads, T, c->num_sms, &pl);
        if (s) return s;
    }
    const uint64_t* ancp = parents ? anc.data() : nullptr;
    s = check_workspace(c, pl, workspace, workspace_bytes);
    if (s) return s;
    if (c->B == 0 || T == 0) {
        return ok();
    }
    s = ensure_device(c);
    if (s) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int64_t* lw = c->lens.data() + static_cast<size_t>(layer) * c->B;
    if (!pl.generic && pl.mt == 1 && max_n > 0 && (pl.R <= tc_min_rows(c) || !tc_capable(c))) {
        // Warps own whole tiles: the attention kernel writes the new rows into
        // the cache itself (one launch instead of two).
        for (int b = 0; b < c->B; ++b) lw[b] += n_new[b];
        bool enqueued = false;
        s = do_attention(c, layer, q, pl, n_new, out, workspace, workspace_bytes, st, k_new, v_new, &enqueued, ancp);
        if (s && !enqueued)
            for (int b = 0; b < c->B; ++b) lw[b] -= n_new[b];  // nothing ran: lengths unchanged
        return s;
    }
    s = do_append(c, layer, k_new, v_new, T, n_new, max_n, st);
    if (s) return s;
    for (int b = 0; b < c->B; ++b) lw[b] += n_new[b];
    s = do_attention(c, layer, q, pl, n_new, out, workspace, workspace_bytes, st, nullptr, nullptr, nullptr, ancp);
    if (s) {
        // The append already ran on the stream; its lengths stand.
        return s;
    }
    return ok();
}

kvc_status kvc_gqa_attention(kvc_cache* c, int layer, const void* q, int q_heads, int T, const int32_t* n_new,
                             void* out, void* workspace, size_t workspace_bytes, void* stream) {
    return gqa_attention_impl(c, layer, q, q_heads, T, n_new, nullptr, out, workspace, workspace_bytes, stream);
}

kvc_status kvc_gqa_attention_tree(kvc_cache* c, int layer, const void* q, int q_heads, int T, const int32_t* n_new,
                                  const int32_t* parents, void* out, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    if (c && c->B > 0 && !parents) return fail(KVC_ERR_ARG, "parents is null");
    return gqa_attention_impl(c, layer, q, q_heads, T, n_new, parents, out, workspace, workspace_bytes, stream);
}

kvc_status kvc_append_attention(kvc_cache* c, int layer, const void* q, const void* k_new, const void* v_new,
                                int q_heads, int T, const int32_t* n_new, void* out, void* workspace,
                                size_t workspace_bytes, void* stream) {
    return append_attention_impl(c, layer, q, k_new, v_new, q_heads, T, n_new, nullptr, out, workspace,
                                 workspace_bytes, stream);
}

kvc_status kvc_append_attention_tree(kvc_cache* c, int layer, const void* q, const void* k_new, const void* v_new,
                                     int q_heads, int T, const int32_t* n_new, const int32_t* parents, void* out,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    if (c && c->B > 0 && !parents) return fail(KVC_ERR_ARG, "parents is null");
    return append_attention_impl(c, layer, q, k_new, v_new, q_heads, T, n_new, parents, out, workspace,
                                 workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Host-buffer form of append + attention
// ---------------------------------------------------------------------------

kvc_status kvc_append_attention_host(kvc_cache* c, int layer, const void* q_host, const void* k_host,
                                     const void* v_host, int q_heads, int T, const int32_t* n_new, void* out_host,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    if (!c) return fail(KVC_ERR_ARG, "handle is null");
    // Everything the device call checks, checked here first on the host
    // pointers (null, 16-byte alignment, shapes, lengths): an error enqueues
    // nothing and reads none of the host buffers.
    kvc_status s = check_host_lens(c);
    if (s) return s;
    int max_n = 0;
    s = validate_append(c, layer, k_host, v_host, T, n_new, &max_n);
    if (s) return s;
    std::vector<int64_t> after(c->B);
    const int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    for (int b = 0; b < c->B; ++b) after[b] = lens[b] + n_new[b];
    AttnPlan pl;
    s = validate_attention(c, layer, q_host, q_heads, T, n_new, out_host, after.data(), &pl, 0);
    if (s) return s;
    if (c->B == 0 || T == 0) return ok();
    s = ensure_device(c);
    if (s) return s;
    s = plan_shape(c, q_heads, T, c->num_sms, &pl);
    if (s) return s;
    s = check_workspace(c, pl, workspace, workspace_bytes);
    if (s) return s;

    const size_t row = static_cast<size_t>(c->d) * io_esize(c);
    const size_t q_bytes = static_cast<size_t>(c->B) * q_heads * T * row;
    const size_t kv_bytes = static_cast<size_t>(c->B) * c->Hkv * T * row;
    const size_t off_k = round256(q_bytes), off_v = off_k + round256(kv_bytes), off_o = off_v + round256(kv_bytes);
    s = ensure_host_staging(c, off_o + round256(q_bytes));
    if (s) return s;
    kvc_cache::HostSlot& hs = c->hslot[c->hnext];
    char* dev = static_cast<char*>(hs.buf);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Inputs into this slot once the last call that read it has computed.
    cudaError_t e = cudaStreamWaitEvent(c->h2d, hs.computed, 0);
    if (e == cudaSuccess) e = copy_chunk(dev, q_host, c->B, q_heads, T, row, n_new, cudaMemcpyHostToDevice, c->h2d);
    if (e == cudaSuccess)
        e = copy_chunk(dev + off_k, k_host, c->B, c->Hkv, T, row, n_new, cudaMemcpyHostToDevice, c->h2d);
    if (e == cudaSuccess)
        e = copy_chunk(dev + off_v, v_host, c->B, c->Hkv, T, row, n_new, cudaMemcpyHostToDevice, c->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(hs.in_ready, c->h2d);
    // The step waits for its inputs and for the slot's previous output to have left.
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hs.in_ready, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hs.out_done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "host-call input copies");
    c->hnext ^= 1;
    s = append_attention_impl(c, layer, dev, dev + off_k, dev + off_v, q_heads, T, n_new, nullptr, dev + off_o,
                              workspace, workspace_bytes, stream);
    if (s) return s;
    e = cudaEventRecord(hs.computed, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->d2h, hs.computed, 0);
    if (e == cudaSuccess)
        e = copy_chunk(out_host, dev + off_o, c->B, q_heads, T, row, n_new, cudaMemcpyDeviceToHost, c->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(hs.out_done, c->d2h);
    if (e != cudaSuccess) return cuda_fail(e, "host-call output copy");
    return ok();
}

kvc_status kvc_host_copies_done(kvc_cache* c, void* stream) {
    if (!c) return fail(KVC_ERR_ARG, "handle is null");
    if (!c->h2d) return ok();  // no host-buffer call yet
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    for (auto& hs : c->hslot)
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hs.out_done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "host-call completion wait");
    return ok();
}

kvc_status kvc_length(const kvc_cache* c, int64_t* out) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    if (!c || !out) return fail(KVC_ERR_ARG, "null argument");
    for (int l = 1; l < c->layers; ++l)
        for (int b = 0; b < c->B; ++b)
            if (c->lens[static_cast<size_t>(l) * c->B + b] != c->lens[b])
                return fail(KVC_ERR_LAYER_MISMATCH,
                            "a forward pass stopped part-way: layer %d row %d has %lld tokens, layer 0 has %lld", l, b,
                            static_cast<long long>(c->lens[static_cast<size_t>(l) * c->B + b]),
                            static_cast<long long>(c->lens[b]));
    for (int b = 0; b < c->B; ++b) out[b] = c->lens[b];
    return ok();
}

kvc_status kvc_truncate(kvc_cache* c, const int64_t* new_lens) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    if (!c) return fail(KVC_ERR_ARG, "null cache handle");
    if (c->B > 0 && !new_lens) return fail(KVC_ERR_ARG, "new_lens is null");
    std::vector<int64_t> cur(c->B);
    kvc_status s = kvc_length(c, cur.data());
    if (s) return s;
    for (int b = 0; b < c->B; ++b) {
        if (new_lens[b] < 0 || new_lens[b] > cur[b])
            return fail(KVC_ERR_ARG, "row %d: invalid truncation length %lld (length %lld)", b,
                        static_cast<long long>(new_lens[b]), static_cast<long long>(cur[b]));
        // A ring still holds positions cur - max_len .. cur - 1; the keys a
        // query after the truncation may need, new - window + 1 .. new - 1,
        // must be among them (nothing is needed after a truncation to 0).
        if (c->ring && new_lens[b] > 0 &&
            std::max<int64_t>(0, new_lens[b] - c->window + 1) < cur[b] - c->max_len)
            return fail(KVC_ERR_ARG, "row %d: a ring cache cannot go back to %lld from %lld", b,
                        static_cast<long long>(new_lens[b]), static_cast<long long>(cur[b]));
    }
    for (int l = 0; l < c->layers; ++l)
        for (int b = 0; b < c->B; ++b) c->lens[static_cast<size_t>(l) * c->B + b] = new_lens[b];
    return ok();
}

kvc_status kvc_reset(kvc_cache* c) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    if (!c) return fail(KVC_ERR_ARG, "null cache handle");
    std::fill(c->lens.begin(), c->lens.end(), 0);
    return ok();
}

kvc_status kvc_set_lens(kvc_cache* c, int layer, const int64_t* lens) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    kvc_status s = check_layer(c, layer);
    if (s) return s;
    if (!lens && c->B > 0) return fail(KVC_ERR_ARG, "lens is null");
    const int64_t top = c->ring ? 0x7fffffffll - c->max_len : c->max_len;  // a ring counts every position
    for (int b = 0; b < c->B; ++b)
        if (lens[b] < 0 || lens[b] > top)
            return fail(KVC_ERR_ARG, "row %d: length %lld outside 0..%lld", b, static_cast<long long>(lens[b]),
                        static_cast<long long>(top));
    for (int b = 0; b < c->B; ++b) c->lens[static_cast<size_t>(layer) * c->B + b] = lens[b];
    return ok();
}

kvc_status kvc_get_lens(const kvc_cache* c, int layer, int64_t* out) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    kvc_status s = check_layer(c, layer);
    if (s) return s;
    if (!out && c->B > 0) return fail(KVC_ERR_ARG, "out is null");
    for (int b = 0; b < c->B; ++b) out[b] = c->lens[static_cast<size_t>(layer) * c->B + b];
    return ok();
}

kvc_status kvc_device_status(kvc_cache* c, void* workspace, void* stream, int32_t* code) {
    if (!c || !workspace || !code) return fail(KVC_ERR_ARG, "null argument");
    kvc_status s = read_error_word(workspace, static_cast<cudaStream_t>(stream), code);
    // After an error, make the next call on this handle clear the workspace header again.
    if (*code != 0) c->last_ws = nullptr;
    return s;
}

kvc_status kvc_selftest_bounded_wait(void* workspace, uint64_t limit_ns, void* stream) {
    if (!workspace) return fail(KVC_ERR_ARG, "workspace is null");
    cudaError_t e = launch_wait_selftest(static_cast<int*>(workspace), limit_ns, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return ok();
}

kvc_status kvc_set_window(kvc_cache* c, int window, int ring) {
    if (!c) return fail(KVC_ERR_ARG, "null cache handle");
    kvc_status s = check_host_lens(c);
    if (s) return s;
    if (window < 0) return fail(KVC_ERR_ARG, "window = %d < 0", window);
    if (ring != 0 && ring != 1) return fail(KVC_ERR_ARG, "ring must be 0 or 1");
    if (ring) {
        if (c->pg.table) return fail(KVC_ERR_ARG, "a paged cache cannot also be a ring");
        if (window < 1 || window > c->max_len) return fail(KVC_ERR_ARG, "a ring cache needs a window of 1..max_len");
        // the largest key tile any kernel of this cache reads
        const int tile = tc_capable(c) ? 128 : key_tile_keys(c->d, c->dtype == KVC_FP8_E4M3);
        if (!generic_path(c) && c->max_len % tile != 0)
            return fail(KVC_ERR_ARG, "this ring cache needs max_len %% %d == 0 (key tiles never wrap)", tile);
    }
    if ((ring != 0) != c->ring)
        for (int64_t L : c->lens)
            if (L != 0) return fail(KVC_ERR_ARG, "ring storage can only change on an empty cache");
    c->window = window;
    c->ring = ring != 0;
    return ok();
}

size_t kvc_device_lens_bytes(const kvc_cache* c) {
    return c ? static_cast<size_t>(c->layers) * c->B * sizeof(int32_t) : 0;
}

kvc_status kvc_lens_to_device(kvc_cache* c, int32_t* dev_lens, void* stream) {
    if (!c) return fail(KVC_ERR_ARG, "null cache handle");
    if (c->lens_on_device) return fail(KVC_ERR_ARG, "the lengths are already on the device");
    if (c->B > 0 && !dev_lens) return fail(KVC_ERR_ARG, "dev_lens is null");
    if ((reinterpret_cast<uintptr_t>(dev_lens) & 3u) != 0) return fail(KVC_ERR_ARG, "dev_lens not 4-byte aligned");
    kvc_status s = ensure_device(c);
    if (s) return s;
    std::vector<int32_t> h(c->lens.size());
    for (size_t i = 0; i < h.size(); ++i) h[i] = static_cast<int32_t>(c->lens[i]);
    if (!h.empty()) {
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cudaError_t e = cudaMemcpyAsync(dev_lens, h.data(), h.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // h is local
        if (e != cudaSuccess) return cuda_fail(e, "copying the lengths to the device");
    }
    c->dev_lens = dev_lens;
    c->lens_on_device = true;
    return ok();
}

kvc_status kvc_lens_from_device(kvc_cache* c, void* stream) {
    if (!c) return fail(KVC_ERR_ARG, "null cache handle");
    if (!c->lens_on_device) return fail(KVC_ERR_ARG, "the lengths are on the host");
    std::vector<int32_t> h(c->lens.size());
    if (!h.empty()) {
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cudaError_t e = cudaMemcpyAsync(h.data(), c->dev_lens, h.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "copying the lengths from the device");
    }
    const int64_t top = c->ring ? 0x7fffffffll - c->max_len : c->max_len;
    for (size_t i = 0; i < h.size(); ++i)
        if (h[i] < 0 || h[i] > top)
            return fail(KVC_ERR_ARG, "device length %d of slot %zu is outside 0..%lld (left on the device)", h[i], i,
                        static_cast<long long>(top));
    for (size_t i = 0; i < h.size(); ++i) c->lens[i] = h[i];
    c->lens_on_device = false;
    c->dev_lens = nullptr;
    return ok();
}

kvc_status kvc_decode_step(kvc_cache* c, int layer, const void* q, const void* k_new, const void* v_new, int q_heads,
                           int T, const int32_t* n_new_dev, void* out, void* workspace, size_t workspace_bytes,
                           void* stream) {
    kvc_status s = check_layer(c, layer);
    if (s) return s;
    if (!c->lens_on_device) return fail(KVC_ERR_ARG, "the lengths are on the host: call kvc_lens_to_device first");
    if (generic_path(c))
        return fail(KVC_ERR_ARG, "device-resident steps serve bf16 and fp8 caches of head_dim %d and bf16 caches of "
                                 "head_dim %d only", kHeadDimBf16, kHeadDimSmall);
    if (c->B == 0 || T == 0) return ok();
    if (T < 0) return fail(KVC_ERR_ARG, "T = %d < 0", T);
    if (!q || !k_new || !v_new || !out || !n_new_dev) return fail(KVC_ERR_ARG, "null pointer argument");
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
        return fail(KVC_ERR_ARG, "q / k_new / v_new / out not 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(n_new_dev) & 3u) != 0) return fail(KVC_ERR_ARG, "n_new not 4-byte aligned");
    s = ensure_device(c);
    if (s) return s;
    AttnPlan pl;
    s = plan_shape(c, q_heads, T, c->num_sms, &pl);
    if (s) return s;
    if (pl.mt != 1)
        return fail(KVC_ERR_SHAPE, "device-resident steps take G * T <= 16 query rows per KV head (G * T = %d)",
                    pl.R);
    if (static_cast<long long>(pl.NB) * ((c->max_len + kKeyTile - 1) / kKeyTile) * c->Hkv > 0x7fffffffll)
        return fail(KVC_ERR_ARG, "too many key tiles for one call");
    s = check_workspace(c, pl, workspace, workspace_bytes);
    if (s) return s;
    s = encode_layer_maps(c, layer);
    if (s) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    if (workspace != c->last_ws) {
        cudaError_t e = cudaMemsetAsync(workspace, 0, pl.ws_err, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
        c->last_ws = workspace;
    }
    DevicePlan* plan = reinterpret_cast<DevicePlan*>(wsb + pl.ws_err);
    const int grid = c->num_sms;

    PlanParams pp;
    pp.n_new = n_new_dev;
    pp.lens = c->dev_lens + static_cast<size_t>(layer) * c->B;
    pp.plan = plan;
    pp.err = reinterpret_cast<int*>(wsb);
    pp.B = c->B;
    pp.T = T;
    pp.R = pl.R;
    pp.RPB = pl.RPB;
    pp.RB = pl.RB;
    pp.NB = pl.NB;
    pp.Hkv = c->Hkv;
    pp.num_ctas = grid;
    pp.max_len = c->max_len;
    pp.window = c->window;
    pp.ring = c->ring ? 1 : 0;
    pp.key_tile = key_tile_keys(c->d, c->dtype == KVC_FP8_E4M3);
    cudaError_t e = launch_decode_plan(pp, st);
    if (e != cudaSuccess) return cuda_fail(e, "device plan launch");
    ++c->launches;

    static_assert(sizeof(DecodeParams) < 32000, "kernel parameter block too large");
    DecodeParams p{};
    p.dplan = plan;
    p.err = reinterpret_cast<int*>(wsb);
    p.partials = reinterpret_cast<float*>(wsb + pl.ws_err + pl.ws_plan);
    p.q = q;
    p.out = out;
    p.B = c->B;
    p.Hq = pl.Hq;
    p.Hkv = c->Hkv;
    p.G = pl.G;
    p.T = pl.T;
    p.max_len = c->max_len;
    p.R = pl.R;
    p.RPB = pl.RPB;
    p.RB = pl.RB;
    p.NB = pl.NB;
    p.part_rows = pl.part_rows;
    p.num_ctas = grid;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(c->d)));
    p.append_new = 1;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = c->k[layer];
    p.v_cache = c->v[layer];
    p.Tn = T;
    p.window = c->window;
    p.ring = c->ring ? 1 : 0;
    p.pg = c->pg;
    set_decode_scales(c, layer, &p);
    e = launch_decode_bf16(p, c->tmK[layer], c->tmV[layer], 1, grid, c->dtype == KVC_FP8_E4M3, c->d, st);
    if (e != cudaSuccess) return cuda_fail(e, "split-KV attention launch");
    ++c->launches;

    static_assert(sizeof(CombineParams) < 32000, "kernel parameter block too large");
    CombineParams cp{};
    cp.dplan = plan;
    cp.partials = p.partials;
    cp.out = out;
    cp.d = c->d;
    cp.Hq = pl.Hq;
    cp.Hkv = c->Hkv;
    cp.G = pl.G;
    cp.T = pl.T;
    cp.R = pl.R;
    cp.RPB = pl.RPB;
    cp.RB = pl.RB;
    cp.NB = pl.NB;
    cp.ways = pl.ways;
    cp.part_rows = pl.part_rows;
    cp.num_ctas = grid;
    e = launch_combine_bf16(cp, st);
    if (e != cudaSuccess) return cuda_fail(e, "split-KV combine launch");
    ++c->launches;
    return ok();
}

uint64_t kvc_kernel_launches(const kvc_cache* c) { return c ? c->launches : 0; }

const char* kvc_last_error(void) { return g_last_error.c_str(); }

const char* kvc_version(void) { return "kvc 0.1 (sm_103a)"; }

}  // extern "C"

// ===========================================================================
// Allocation-free attention (kvc_gqa_attention_noalloc)
//
// For callers that cannot allocate device memory themselves: the split-KV
// scratch (header and partial results) lives in one
// file-scope device array instead of a caller-provided workspace.  The array
// is part of this library's device image, so every GPU that loads the
// library holds its KVC_NOALLOC_SCRATCH_BYTES until the process exits.
// ===========================================================================

static __device__ __align__(256) unsigned char kvc_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name only stands for the symbol; the address a kernel can use
// comes from cudaGetSymbolAddress, looked up once per device with that
// device current and cached.
kvc_status noalloc_scratch_address(int device, void** out) {
    if (device < 0 || device >= kNoAllocMaxDevices) return fail(KVC_ERR_ARG, "device %d out of range", device);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[device]) {
        void* addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, kvc_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_noalloc_addr[device] = addr;
    }
    *out = g_noalloc_addr[device];
    return ok();
}

}  // namespace

extern "C" kvc_status kvc_gqa_attention_noalloc(kvc_cache* c, int layer, const void* q, int q_heads, int T,
                                                const int32_t* n_new, void* out, void* stream) {
    kvc_status s0 = check_host_lens(c);
    if (s0) return s0;
    kvc_status s = check_layer(c, layer);
    if (s) return s;
    if (generic_path(c))
        return fail(KVC_ERR_ARG, "the allocation-free variant serves bf16 and fp8 caches of head_dim %d and bf16 "
                                 "caches of head_dim %d only", kHeadDimBf16, kHeadDimSmall);
    AttnPlan pl;
    const int64_t* lens = c->lens.data() + static_cast<size_t>(layer) * c->B;
    s = validate_attention(c, layer, q, q_heads, T, n_new, out, lens, &pl, 0);
    if (s) return s;
    if (c->B == 0 || T == 0) return ok();
    s = ensure_device(c);
    if (s) return s;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != c->device) return fail(KVC_ERR_ARG, "current device %d is not the cache's device %d", dev, c->device);
    s = plan_shape(c, q_heads, T, c->num_sms, &pl);
    if (s) return s;
    if (pl.generic)
        return fail(KVC_ERR_ARG, "the allocation-free variant takes at most 64 query rows per KV head on a cache of "
                                 "head_dim %d (G * T = %d)", kHeadDimSmall, pl.R);
    if (pl.ws_min > static_cast<size_t>(KVC_NOALLOC_SCRATCH_BYTES))
        return fail(KVC_ERR_WORKSPACE, "this call needs %zu bytes of scratch; the static scratch holds %zu",
                    pl.ws_min, static_cast<size_t>(KVC_NOALLOC_SCRATCH_BYTES));
    void* scratch = nullptr;
    s = noalloc_scratch_address(dev, &scratch);
    if (s) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left: zero the header after
    // the error word (the counters), the part the kernels need to start at
    // zero.  The error word is left alone, so an error stays recorded until
    // kvc_noalloc_status reads and clears it.
    e = cudaMemsetAsync(static_cast<uint8_t*>(scratch) + sizeof(int), 0, pl.ws_err - sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch)");
    c->last_ws = scratch;
    return do_attention(c, layer, q, pl, n_new, out, scratch, KVC_NOALLOC_SCRATCH_BYTES, st);
}

extern "C" kvc_status kvc_noalloc_status(void* stream, int32_t* code) {
    if (!code) return fail(KVC_ERR_ARG, "null argument");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    void* scratch = nullptr;
    kvc_status s = noalloc_scratch_address(dev, &scratch);
    if (s) return s;
    return read_error_word(scratch, static_cast<cudaStream_t>(stream), code);
}
