// Internal declarations shared by the host library and the kernels of libkvc.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc.h"

namespace kvc {

constexpr int kMaxBatch = KVC_MAX_BATCH;
constexpr int kMaxGroups = 1024;  // (row, row-block) groups of one attention call
constexpr int kMaxCtas = 1024;    // attention CTAs (one per SM)
constexpr int kMaxTreeQueries = 1024;  // B * T of a tree-verify call (one ancestor mask per query)

// Paged storage: a row's logical position a lives at page table[b * mpr + a / page],
// offset a % page, of buffers shaped [num_pages, Hkv, page, d]; table null:
// contiguous [B, Hkv, max_len, d] (or a ring).  Row index of the 2-D
// (rows x d) view of the buffer, for (row b, KV head kvh, position a); *bad is
// set for an entry outside 0 .. num_pages - 1, whose row is then page 0's.
struct Paging {
    const int32_t* table;
    int page, mpr, num_pages;
};
__host__ __device__ __forceinline__ int phys_row(const Paging& pg, int ring, int Hkv, int max_len, int b, int kvh,
                                                 int a, bool* bad) {
    if (pg.table) {
        const int e = pg.table[b * pg.mpr + a / pg.page];
        const bool ok = e >= 0 && e < pg.num_pages;
        if (!ok) *bad = true;
        return ((ok ? e : 0) * Hkv + kvh) * pg.page + a % pg.page;
    }
    return (b * Hkv + kvh) * max_len + (ring ? a % max_len : a);
}

// Keys per K/V tile of the split-KV kernel for 128-wide heads (see
// key_tile_keys), and the head width the TMA / tensor-core kernels are built
// for (the split-KV kernel also takes bf16 storage of head width kHeadDimSmall).
constexpr int kKeyTile = 64;
constexpr int kHeadDimBf16 = 128;
constexpr int kHeadDimSmall = 64;
// Keys per split-KV tile: 64, or 128 for bf16 storage of head width
// kHeadDimSmall and for FP8 storage (a 64-key tile there would carry half the
// bytes of a bf16 128-wide one for the same per-tile work).
__host__ __device__ constexpr int key_tile_keys(int d, bool fp8) {
    return ((d == kHeadDimSmall && !fp8) || fp8) ? 2 * kKeyTile : kKeyTile;
}
// FP8 E4M3 caches: one K and one V scale per KV head (at most this many heads).
constexpr int kMaxScaleHeads = 64;

// ---------------------------------------------------------------------------
// In-place append: k_new/v_new [B, Hkv, T, d] -> cache rows lens[b] .. lens[b]+n_new[b]-1.
// ---------------------------------------------------------------------------
struct AppendParams {
    const uint8_t* k_new;
    const uint8_t* v_new;
    uint8_t* k_cache;
    uint8_t* v_cache;
    int B, Hkv, T, max_len;
    int row_bytes;  // d * element size, a multiple of 16
    int ring;       // slots are positions mod max_len
    Paging pg;
    // FP8 E4M3 cache: k_new / v_new rows are bf16 (row_bytes = 2 * d) and are
    // stored as E4M3 codes of x * (1/scale) (d bytes a row).
    int fp8;
    float kscale[kMaxScaleHeads];
    float vscale[kMaxScaleHeads];
    int lens[kMaxBatch];
    int n_new[kMaxBatch];
};

cudaError_t launch_append(const AppendParams& p, int max_n_new, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Split-KV attention (bf16 storage, fp32 accumulation).
//
// Rows.  For one KV head the G*T query rows are r = g*T + t (query head
// kvh*G + g, query t).  Rows are cut into row blocks of RPB = 16*MT rows.
// A "group" is one (b, row block); a "unit" is one (group, kvh); unit
// u = group*Hkv + kvh.  A unit's keys are 0 .. E-1 where E is one past the
// largest visible key of its valid rows; it has nt = ceil(E / 64) tiles.
// Tiles are numbered unit after unit: group q's units own tiles
// gstart[q] .. gstart[q+1]-1, kvh after kvh.  CTA i of P processes tiles
// floor(i*N/P) .. floor((i+1)*N/P)-1, so every CTA gets the same number of
// tiles (+-1) whatever the row lengths.  A unit seen in full by one writer is
// written to `out` directly; otherwise each writer (a CTA, or with warps
// owning whole tiles a warp of it) leaves its partial softmax state in
// sub-slot (u + i) * ways + w, where i is the CTA (u + i is unique per
// (unit, CTA) pair: along the unit/CTA staircase every step raises it), and
// the combine kernel merges them.
// ---------------------------------------------------------------------------
// Per-step plan of the split-KV kernels computed on the device from
// device-resident lengths (graph-capturable steps): the fields the host
// planner otherwise puts in DecodeParams / CombineParams.
struct DevicePlan {
    int skip;         // the step was rejected (a row would overflow): nothing runs
    int total_tiles;
    int prior[kMaxBatch];
    int n_new[kMaxBatch];
    int gstart[kMaxGroups + 1];
    int cta_start[kMaxCtas + 1];
};

struct PlanParams {
    const int32_t* n_new;  // device [B]
    int32_t* lens;         // device [B]: this layer's lengths, advanced by n_new
    DevicePlan* plan;
    int* err;
    int B, T, R, RPB, RB, NB, Hkv, num_ctas, max_len;
    int window, ring;
    int key_tile;  // keys per tile of the split-KV kernel this plan feeds
};

cudaError_t launch_decode_plan(const PlanParams& p, cudaStream_t stream);

struct DecodeParams {
    const DevicePlan* dplan;  // when set, prior / n_new / gstart / total_tiles come from it
    const void* q;      // [B, Hq, T, d] bf16
    void* out;          // [B, Hq, T, d] bf16
    float* partials;    // [(units + P) * ways sub-slots][part_rows][d + 4] : O (d), m, l, pad
    int* err;           // device error word
    int B, Hq, Hkv, G, T, max_len;
    int R, RPB, RB, NB;
    int part_rows;      // rows stored per partial sub-slot: min(R, RPB)
    int total_tiles;
    int num_ctas;
    float scale_log2;   // log2(e) / sqrt(d)
    // In-kernel append (warps owning whole tiles only): when append_new is set
    // the chunk's rows k_new/v_new [B, Hkv, Tn, d] are written to the layer's
    // cache at positions prior[b] .. prior[b]+n_new[b]-1 by the warp that
    // processes the tile holding them, which also patches them into its
    // staged tile, so the append needs no launch of its own.
    const void* k_new;
    const void* v_new;
    void* k_cache;
    void* v_cache;
    int append_new;
    int Tn;
    // Sliding window (0 = none): a query at position p sees keys p - window < a <= p.
    // Ring storage: the key at position a lives in slot a mod max_len.
    int window, ring;
    // Tree verify: query t of row b sees the chunk's tokens u with bit u of
    // anc[b * T + t] set (its path to the root), besides every key before the
    // chunk.  anc is device memory (the workspace); null without a tree.
    const uint64_t* anc;
    Paging pg;
    // FP8 E4M3 cache (kernel variant F8): K of head h reads code * kscale[h],
    // V reads code * vscale[h]; appended rows are quantized with 1/scale.
    float kscale[kMaxScaleHeads];
    float vscale[kMaxScaleHeads];
    int prior[kMaxBatch];    // lens[b] - n_new[b]
    int n_new[kMaxBatch];
    int gstart[kMaxGroups + 1];
};

// Log-sum-exp merge of the units the attention kernel left as partials (one
// CTA per unit; the grid covers every unit and the ones written in full
// return at once).  Partial rows live at
// ((u + cta) * ways + warp) * part_rows + row.
struct CombineParams {
    const DevicePlan* dplan;  // when set, n_new / gstart / cta_start / total_tiles come from it
    const float* partials;
    void* out;
    int d;  // head dimension: 128 or 64
    int Hq, Hkv, G, T, R, RPB, RB, NB;
    int ways;       // partial sub-slots per (unit, CTA)
    int part_rows;  // rows stored per partial sub-slot
    int total_tiles, num_ctas;
    int n_new[kMaxBatch];
    int gstart[kMaxGroups + 1];
    int cta_start[kMaxCtas + 1];  // first tile of each attention CTA: floor(i * N / P)
};

cudaError_t launch_combine_bf16(const CombineParams& p, cudaStream_t stream);

// Grid / block / shared memory of the split-KV kernel for a given MT.
struct DecodeLaunch {
    int mt;
    int threads;
    size_t smem_bytes;
    int ways;  // partial sub-slots per (unit, CTA): 4 when warps own whole tiles
};
// d: the head dimension (128 for bf16 and FP8 storage, or 64 for bf16).
DecodeLaunch decode_launch_shape(int mt, bool fp8, int d);

cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int mt,
                               int grid, bool fp8, int d, cudaStream_t stream);

// ---------------------------------------------------------------------------
// f32 attention (any d <= 256, d % 4 == 0): one CTA per (16-row block, kvh, b),
// all keys of the unit, output written directly; no workspace.
// ---------------------------------------------------------------------------
struct F32Params {
    // kind 0: fp32 storage, queries and outputs; 1: bf16 throughout; 2: FP8
    // E4M3 codes (value = code * kscale / vscale of the KV head), bf16
    // queries and outputs.
    const void* q;
    const void* k_cache;
    const void* v_cache;
    void* out;
    int kind;
    float kscale[kMaxScaleHeads];
    float vscale[kMaxScaleHeads];
    int B, Hq, Hkv, G, T, max_len, d;
    int R;
    int window, ring;  // sliding window (0 = none) and ring storage, as in DecodeParams
    int tree;          // ancestor masks in anc, as in DecodeParams
    Paging pg;
    float scale;  // 1 / sqrt(d)
    // Key-range split: `splits` CTAs per (row block, KV head, row); with more
    // than one, each leaves (m, l, O) of its 16 rows in partials
    // [unit][split][16][d + 2] and the last to arrive (counters[unit]) merges.
    int splits;
    float* partials;
    int* counters;
    int prior[kMaxBatch];
    int n_new[kMaxBatch];
    uint64_t anc[kMaxTreeQueries];
};

constexpr int kGenericMaxSplits = 16;
cudaError_t launch_attn_f32(const F32Params& p, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Attention on tcgen05 (bf16, d = 128) for many query rows per KV head.  One
// CTA per piece of an item; items are packed as
// ((b * Hkv + kvh) * ntb + tb) * npair + pair.  An item's query rows form up to
// two 128-row tiles that share every K/V tile:
//   mode 0 (chunked prefill, T >= 128): tile i = 128 positions tb*128 .. of
//          query head kvh*G + 2*pair + i;
//   mode 1 (packed, T < 128, G*T > 128): tile i = packed rows
//          (2*pair + i)*128 .. of the KV head, row r = g*T + t (ntb = 1);
//   mode 2 (packed, G*T <= 128): one tile of packed rows; the two TMEM S/O
//          buffers and softmax warpgroups take alternate key tiles and their
//          states are merged at the end (ntb = npair = 1).
// ---------------------------------------------------------------------------
constexpr int kMaxPrefillPieces = 1920;
constexpr int kPrefillNoSlot = 0xFFF;   // piece covers all keys of its block: write out directly
constexpr int kMaxPrefillSlots = 4095;  // key-split pieces per launch (each has a partial slot)
// Workspace header: the error word, then one merge counter per (first slot of
// a split block, head); the partials follow the header.
constexpr size_t kWsCounterOffset = 256;
constexpr size_t kWsHeaderBytes = kWsCounterOffset + static_cast<size_t>(kMaxPrefillSlots + 1) * 2 * sizeof(int);
struct PrefillParams {
    const void* q;
    void* out;
    int* err;         // workspace start: error word, merge counters
    float* partials;  // [slot][2 heads][128 rows][d + 4]: O (d), m, l, pad
    int B, Hq, Hkv, G, T, max_len;
    int ntb, npair, n_pieces;
    int mode;          // 0 positions, 1 packed rows in tile pairs, 2 one packed tile (see above)
    int fp8;           // FP8 E4M3 cache: K of head h reads code * kscale[h], V code * vscale[h]
    float kscale[kMaxScaleHeads];
    float vscale[kMaxScaleHeads];
    int window, ring;  // sliding window (0 = none) and ring storage, as in DecodeParams
    Paging pg;
    float scale_log2;
    int prior[kMaxBatch];
    int n_new[kMaxBatch];
    // One CTA per piece, in launch order.
    uint32_t piece_code[kMaxPrefillPieces];   // packed (b, kvh, tb, pair)
    uint32_t piece_tiles[kMaxPrefillPieces];  // key tiles lo | hi << 16 (tiles of 128 keys)
    // slot | index of the piece within its block << 12 | pieces of the block << 22
    // (slot = kPrefillNoSlot when the piece covers all keys of its block)
    uint32_t piece_aux[kMaxPrefillPieces];
};

size_t prefill_smem_bytes();
cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                              const CUtensorMap& tmV, cudaStream_t stream);

// Device error codes written to the workspace error word.
enum DeviceError : int {
    kDevOk = 0,
    kDevTimeoutFull = 1,   // consumer gave up waiting for a K/V tile
    kDevTimeoutEmpty = 2,  // producer gave up waiting for a free stage
    kDevTimeoutDrain = 3,  // abort path gave up waiting for copies in flight
    kDevTimeoutTest = 4,   // the self-test wait expired, as it is meant to
    kDevTimeoutTag = 5,    // consumer gave up waiting for the producer to claim a stage
    kDevOverflow = 6,      // a device-resident step was rejected: a row would pass max_len
    kDevBadPage = 7        // a block-table entry outside 0 .. num_pages - 1 was met (not read / written)
};

// Self-test of the bounded wait: waits on an mbarrier that nothing arrives at,
// for at most `limit_ns`, then records kDevTimeoutTest in *err.
cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace kvc
