// GQA attention on the 5th-generation tensor cores (tcgen05 + TMEM), bf16,
// d = 128, for calls with more than 12 query rows per KV head: chunked
// prefill, speculative verify with large G*T.
//
// What it computes ("Implement grouped-query attention over a preallocated KV
// cache...", "A strong answer", gqa_attention): query t < n_new[b] of head h
// sits at position prior[b] + t (prior = lens - n_new) and attends to keys
// 0 .. prior[b] + t of KV head h / G with softmax scale 1/sqrt(d).  Padded
// queries (t >= n_new[b]) give 0.  QK^T and PV are 128 x 128 x 128 MMAs.
//
// A work item's query rows form up to two 128-row tiles that share every K/V
// tile staged in shared memory (each 64 KB K/V tile then feeds four
// 128x128x128 MMAs):
//   mode 0 (T >= 128): 128 positions of a pair of query heads of the group;
//   mode 1 (T < 128): 128-row tiles of the G*T rows r = g*T + t of one KV
//          head, packed (in [B, Hq, T, d] they are consecutive rows);
//   mode 2 (G*T <= 128): one packed tile; the two TMEM S/O buffers and the two
//          softmax warpgroups take alternate key tiles, so one buffer's softmax
//          runs under the other's MMAs, and the two states are merged at the end.
// Items are launched longest first (the host sorts them by key-tile count).
//
// FP8 E4M3 caches ("16. Prefill, decode and the KV cache", exercise 4): each
// 128-key tile arrives as 128 x 128 bytes in the second half of its stage;
// warps 2 and 3 convert it in place to the f16 tile (and the queries from bf16
// to f16 once), and the MMAs run kind::f16 on f16 operands; the K scale folds
// into the softmax scale and the V scale into the output normalisation.
//
// Warp roles (12 warps):
//   warp 0      TMA producer: Q tiles once, then K and V tiles (128 keys) into
//               two-stage rings guarded by mbarriers.
//   warp 1      MMA issuer (one lane): S_i = Q_i K^T into TMEM, then, once the
//               softmax has written P_i into TMEM over S_i, O_i += P_i V with
//               P_i as the TMEM A operand.  Issue order S0(j), S1(j), PV0(j),
//               S0(j+1), PV1(j), S1(j+1), ... keeps the tensor core busy while
//               each softmax warpgroup works on the other head's tile.
//   warps 4-7   softmax of row tile 0 (mode 2: even key tiles), one thread per query row
//   warps 8-11  softmax of row tile 1 (mode 2: odd key tiles)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).
//
// Softmax is online in base 2 (log2(e)/sqrt(d) folded into one scale) with a
// lazy rescale: the running max used for the exponentials only moves when
// the row max exceeds it by more than 8 (a factor 256), and only then is O
// rescaled in TMEM; O and l share the same reference, so the result is exact.
// Causal mask ("Write the causal mask for a decode step...", bottom-right):
// key tiles past the block's last visible key are never loaded; tiles fully
// visible to every row of the block skip the mask; the rest mask per element
// with a select.  V rows past the last visible key are cleared in shared
// memory before PV, so stale or NaN cache slots never meet p = 0.
// Sliding window and ring storage (same page, "A strong answer", last
// paragraph): with a window W a row sees keys lim - W < a <= lim, tiles before
// the window of the block's first query are never loaded, tiles fully inside
// every row's window skip the mask, and V rows outside every row's window are
// cleared too; in a ring cache key a lives in slot a mod max_len (max_len a
// multiple of 128, so a tile never wraps).
// Every wait is bounded in time; on expiry an error code is recorded.

#include <math.h>

#include <utility>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kThreadsPF = 384;  // 4 warps (producer, MMA issuer, 2 converters / idle) + 8 softmax warps
constexpr int kD = 128;
constexpr int kBoxBytes = 128 * 128;           // 128 rows x 64 columns x 2 B (one swizzled box)
constexpr int kTile128 = 2 * kBoxBytes;         // 128 rows x 128 columns
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;       // log2 of the largest factor kept unrescaled

// Shared memory map (offsets from the 1024-aligned base).
constexpr int kOffQ = 0;                        // Q0, Q1
constexpr int kOffK = 2 * kTile128;             // K stages 0, 1
constexpr int kOffV = 4 * kTile128;             // V stages 0, 1
constexpr int kOffBar = 6 * kTile128;
// A split piece's epilogue stages head i's 128 x (d + 4) float partial block
// at kOffQ + i * kSplitStageBytes: Q, the K stages and the first 4 KB of V
// stage 0, all idle once that head's last PV product has landed.
constexpr int kSplitStageBytes = 128 * (kD + 4) * 4;
static_assert(2 * kSplitStageBytes <= kOffBar, "split staging fits below the barriers");
// barrier indices
// (FP8 caches: TMA completes the *Raw barriers, the converter warps then arm
// Q / KFull / VFull once the tiles are f16)
constexpr int kBarQ = 0, kBarKFull = 1, kBarKEmpty = 3, kBarVFull = 5, kBarVEmpty = 7, kBarS = 9, kBarP = 11,
              kBarO = 13, kBarQRaw = 15, kBarKRaw = 16, kBarVRaw = 18, kNumBars = 20;
constexpr int kConvThreads = 64;  // warps 2 and 3
constexpr size_t kSmemPF = 1024 + kOffBar + 256;

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    // tcgen05 shared-memory matrix descriptor: start >> 4, leading / stride byte
    // offsets >> 4, fixed 0b001 at bits 46-48, 128-byte swizzle.
    return static_cast<uint64_t>((addr & 0x3FFFF) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 (or f16) A and B, M = N = 128.
__device__ __forceinline__ uint32_t instr_desc(bool b_mn_major, bool f16 = false) {
    const uint32_t ab = f16 ? 0u : ((1u << 7) | (1u << 10));  // A and B format: 0 = f16, 1 = bf16
    return (1u << 4) | ab | (static_cast<uint32_t>(b_mn_major) << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

// FP8 caches: one 128-key tile of E4M3 codes (128 rows x 128 bytes, 128-byte
// swizzle) sits in the second half of a stage; convert it in place to the f16
// tile the MMAs read (two 64-column boxes, 128-byte swizzle).  Each thread
// owns whole rows: it reads its row's 128 bytes before writing the row's
// 256, and no other row is touched, so the in-place order is safe.
__device__ __forceinline__ void convert_e4m3_tile(uint8_t* slot, int ct) {
    for (int r = ct; r < 128; r += kConvThreads) {
        const uint8_t* src = slot + kBoxBytes + r * 128;
        uint4 c8[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) c8[c] = *reinterpret_cast<const uint4*>(src + (((c ^ (r & 7))) << 4));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            // fp8 chunk c = columns 16c .. 16c + 15 -> f16 chunks 2c, 2c + 1
            const uint32_t w[4] = {c8[c].x, c8[c].y, c8[c].z, c8[c].w};
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) ptx::e4m3x4_to_f16x2x2(w[i], h[2 * i], h[2 * i + 1]);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int cc = 2 * c + half;  // f16 chunk of the 256-byte row
                uint8_t* dst = slot + (cc >> 3) * kBoxBytes + r * 128 + ((((cc & 7) ^ (r & 7))) << 4);
                *reinterpret_cast<uint4*>(dst) = make_uint4(h[4 * half], h[4 * half + 1], h[4 * half + 2], h[4 * half + 3]);
            }
        }
    }
}

// bf16 -> f16 in place (same layout): the queries of an FP8 cache's MMAs.
__device__ __forceinline__ void convert_bf16_tiles(uint8_t* base, int bytes, int ct) {
    for (int off = ct * 16; off < bytes; off += kConvThreads * 16) {
        uint4 v = *reinterpret_cast<const uint4*>(base + off);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = ptx::pack_f16x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
        *reinterpret_cast<uint4*>(base + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 64 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Packed fp32 pair arithmetic (two lanes per instruction) and a 3-input max.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// One piece: a key-tile range of one work item (b, KV head, row block, pair).
struct Piece {
    int b, kvh, t0, h0, nh;      // row, KV head; mode 0: first position, first head; row tiles (1 or 2)
    int pr0;                     // modes 1, 2: first packed row of tile 0 (row r = g*T + t of the KV head)
    int prior, nn;               // prior length and new tokens of row b
    int kmax, nkt_all;           // last visible key of the block, its key tiles
    int full_below;              // keys <= this are visible to every valid row of the item
    int kt0, nkt;                // this piece's tiles: kt0 .. kt0 + nkt - 1
    int slot;                    // partial slot, or kPrefillNoSlot
    int kidx, npc;               // index of the piece within its block, pieces of the block
};

__device__ __forceinline__ Piece decode_piece(const PrefillParams& p, int idx) {
    Piece pc;
    int code = static_cast<int>(p.piece_code[idx]);
    const int pair = code % p.npair;
    code /= p.npair;
    const int tb = code % p.ntb;
    code /= p.ntb;
    pc.kvh = code % p.Hkv;
    pc.b = code / p.Hkv;
    pc.prior = p.prior[pc.b];
    pc.nn = p.n_new[pc.b];
    if (p.mode == 0) {
        pc.t0 = tb * 128;
        pc.h0 = pc.kvh * p.G + 2 * pair;
        pc.nh = min(2, p.G - 2 * pair);
        pc.pr0 = 0;
        pc.kmax = pc.prior + min(pc.t0 + 127, pc.nn - 1);
        pc.full_below = pc.prior + pc.t0;
    } else {
        // Packed rows: every valid row has 0 <= t < min(T, nn), so keys up to
        // prior are visible to all of them and prior + min(T, nn) - 1 is the
        // last key any of them sees.
        pc.t0 = 0;
        pc.h0 = pc.kvh * p.G;
        pc.pr0 = 2 * pair * 128;
        pc.nh = (p.mode == 2) ? 1 : min(2, (p.G * p.T - pc.pr0 + 127) / 128);
        pc.kmax = pc.prior + min(p.T, pc.nn) - 1;
        pc.full_below = pc.prior;
    }
    pc.nkt_all = pc.kmax / 128 + 1;
    const uint32_t tiles = p.piece_tiles[idx];
    pc.kt0 = static_cast<int>(tiles & 0xFFFF);
    pc.nkt = static_cast<int>(tiles >> 16) - pc.kt0;
    const uint32_t aux = p.piece_aux[idx];
    pc.slot = static_cast<int>(aux & 0xFFF);
    pc.kidx = static_cast<int>((aux >> 12) & 0x3FF);
    pc.npc = static_cast<int>(aux >> 22);
    return pc;
}

// Epilogue of one piece of a key-split block (head i, row r): leave
// (O, m, l) in the piece's partial slot; the piece that finishes last (a
// counter per block and head) merges all of them:
// o = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k.  Kept out of line so its
// registers do not press on the softmax loop.
//
// `stage` is this head's 128 x (d + 4) float block of shared memory, idle
// once the head's last PV product has landed.  Both directions go through
// it: a row per thread on the shared side (the 4-float pad puts 8
// consecutive rows on distinct banks) and whole 512-byte spans per warp
// instruction on the global side.  The merging piece pulls each other
// piece's block in with cp.async, all of it in flight at once.  tS: this
// head's S columns, idle by now, hold the running sum of O when a block has
// more than two pieces.
__device__ __noinline__ void split_epilogue(float* partials, int* err, uint32_t tS, uint32_t tO, int i, int r, bool valid,
                                            float m_ref, float l, int slot, int kidx, int npc, __nv_bfloat16* dst,
                                            volatile int* merge_flag, float out_scale, float* stage) {
    constexpr int kRowF = kD + 4;             // floats per partial row: O, m, l, pad
    constexpr int kChunks = 128 * kRowF / 4;  // 16-byte chunks of one head's block
    static_assert(kChunks % 128 == 0, "each thread moves the same number of chunks");
    const int slot0 = slot - kidx;
    auto block_of = [&](int sl) { return partials + (static_cast<size_t>(sl) * 2 + i) * 128 * kRowF; };
    float* srow = stage + r * kRowF;
    // The warpgroup may still be reading shared memory that overlaps the
    // staging block (the packed mode's exchange of the odd-tile state).
    ptx::named_barrier_sync(1 + i, 128);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t w[32];
        tmem_ld32(tO + c * 32, w);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<uint4*>(srow + c * 32 + e) = make_uint4(w[e], w[e + 1], w[e + 2], w[e + 3]);
    }
    srow[kD] = m_ref;
    srow[kD + 1] = l;
    ptx::named_barrier_sync(1 + i, 128);
    {
        float4* g = reinterpret_cast<float4*>(block_of(slot));
        const float4* s4 = reinterpret_cast<const float4*>(stage);
#pragma unroll 3
        for (int x = r; x < kChunks; x += 128) g[x] = s4[x];
    }
    __threadfence();
    ptx::named_barrier_sync(1 + i, 128);
    int* counter = err + kWsCounterOffset / sizeof(int) + slot0 * 2 + i;
    if (r == 0) merge_flag[i] = (atomicAdd(counter, 1) == npc - 1) ? 1 : 0;
    ptx::named_barrier_sync(1 + i, 128);
    if (!merge_flag[i]) return;
    __threadfence();
    // The pieces are combined in the fixed order k = 0 .. npc - 1 whichever of
    // them merges, so repeated calls give the same bits.  M and L first: with
    // two pieces the other one is staged now and its (m, l) read from shared
    // memory; with more, each (m, l) comes from its slot.
    const uint32_t sbase = ptx::smem_addr(stage);
    int staged = -1;
    auto stage_piece = [&](int k) {
        ptx::named_barrier_sync(1 + i, 128);  // every row of the previous block has been read
        const float* src = block_of(slot0 + k);
#pragma unroll 3
        for (int x = r; x < kChunks; x += 128) ptx::cp_async_16(sbase + x * 16, src + x * 4);
        ptx::cp_async_wait_all();
        ptx::named_barrier_sync(1 + i, 128);
        staged = k;
    };
    if (npc == 2) stage_piece(1 - kidx);
    auto m_of = [&](int k) {
        return k == kidx ? m_ref : k == staged ? srow[kD] : __ldcg(block_of(slot0 + k) + r * kRowF + kD);
    };
    auto l_of = [&](int k) {
        return k == kidx ? l : k == staged ? srow[kD + 1] : __ldcg(block_of(slot0 + k) + r * kRowF + kD + 1);
    };
    float M = -INFINITY;
    for (int k = 0; k < npc; ++k) M = fmaxf(M, m_of(k));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
    for (int k = 0; k < npc; ++k) {
        const float mk = m_of(k);
        if (mk != -INFINITY) L += l_of(k) * ptx::ex2(mk - Mu);
    }
    const float inv = (valid && L > 0.f) ? out_scale / L : 0.f;  // out_scale: an FP8 cache's V scale
    auto weight = [&](int k) {
        const float mk = m_of(k);
        return (mk == -INFINITY) ? 0.f : ptx::ex2(mk - Mu);
    };
    auto write_out = [&](int c, const float (&acc)[32]) {
        if (!valid) return;
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
            uint4 q4;
            q4.x = ptx::pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
            q4.y = ptx::pack_bf16x2(acc[e + 2] * inv, acc[e + 3] * inv);
            q4.z = ptx::pack_bf16x2(acc[e + 4] * inv, acc[e + 5] * inv);
            q4.w = ptx::pack_bf16x2(acc[e + 6] * inv, acc[e + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + e) = q4;
        }
    };
    if (npc == 2) {
        // o = w_1 O_1 + w_0 O_0 in one pass: the own O from TMEM, the other from
        // its staged block.
        const float w_own = weight(kidx), w_oth = weight(1 - kidx);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t w[32];
            tmem_ld32(tO + c * 32, w);
            tmem_ld_wait();
            float acc[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 o4 = *reinterpret_cast<const float4*>(srow + c * 32 + e);
                const float oth[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float own = __uint_as_float(w[e + u]);
                    acc[e + u] = kidx == 0 ? fmaf(w_oth, oth[u], w_own * own) : fmaf(w_own, own, w_oth * oth[u]);
                }
            }
            write_out(c, acc);
        }
    } else {
        // O = sum_k 2^(m_k - M) O_k, the running sum kept in this head's S
        // columns (idle now) between pieces; the own O_k comes from TMEM, the
        // others from their staged blocks.
        for (int k = 0; k < npc; ++k) {
            const bool own = k == kidx, first = k == 0, last = k == npc - 1;
            if (!own) stage_piece(k);
            const float wk = weight(k);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float ok[32], acc[32];
                uint32_t w[32];
                if (own) {
                    tmem_ld32(tO + c * 32, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) ok[e] = __uint_as_float(w[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 o4 = *reinterpret_cast<const float4*>(srow + c * 32 + e);
                        ok[e] = o4.x, ok[e + 1] = o4.y, ok[e + 2] = o4.z, ok[e + 3] = o4.w;
                    }
                }
                if (first) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = wk * ok[e];
                } else {
                    tmem_ld32(tS + c * 32, w);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = fmaf(wk, ok[e], __uint_as_float(w[e]));
                }
                if (!last) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(acc[e]);
                    tmem_st32(tS + c * 32, w);
                    tmem_st_wait();
                } else {
                    write_out(c, acc);
                }
            }
        }
    }
    if (r == 0) *counter = 0;  // ready for the next call
}

// kWin: the cache has a sliding window (and possibly ring storage); without
// one the window code is compiled out.  kAlt: mode 2 (one packed row tile,
// alternate key tiles per TMEM buffer); modes 0 and 1 otherwise.  kF8: the
// cache holds E4M3 codes (converted to f16 in shared memory by warps 2 and 3;
// the MMAs run on f16 with the queries converted too).
template <bool kWin, bool kAlt, bool kF8>
__global__ void __launch_bounds__(kThreadsPF, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = sbase + kOffBar;
    auto bar = [&](int i) { return bar0 + 8 * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kOffBar + kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + kNumBars * 8 + 8);
    volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + kOffBar + kNumBars * 8 + 16);  // per head

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        const int ready = kF8 ? 2 : 1;  // FP8: both converter warps arrive; else the TMA's arrive
        ptx::mbar_init(bar(kBarQ), ready);
        ptx::mbar_init(bar(kBarQRaw), 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(kBarKFull + s), ready);
            ptx::mbar_init(bar(kBarKRaw + s), 1);
            ptx::mbar_init(bar(kBarVRaw + s), 1);
            ptx::mbar_init(bar(kBarKEmpty + s), 1);
            ptx::mbar_init(bar(kBarVFull + s), ready);
            ptx::mbar_init(bar(kBarVEmpty + s), 1);
            ptx::mbar_init(bar(kBarS + s), 1);
            ptx::mbar_init(bar(kBarP + s), 4);
            ptx::mbar_init(bar(kBarO + s), 1);
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmQ);
        ptx::tma_prefetch_desc(&tmK);
        ptx::tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         sbase + kOffBar + kNumBars * 8)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    ptx::grid_dependency_wait();
    ptx::launch_dependents();

    // Padded queries (t >= n_new[b]) output zeros; spread over the whole grid.
    {
        const int rows_total = p.B * p.Hq * p.T;
        for (int row = blockIdx.x * kThreadsPF + tid; row < rows_total; row += gridDim.x * kThreadsPF) {
            const int t = row % p.T;
            const int b = row / (p.Hq * p.T);
            if (t >= p.n_new[b]) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(row) * kD);
#pragma unroll
                for (int i = 0; i < kD * 2 / 16; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }

    const Piece pc = decode_piece(p, blockIdx.x);
    const int b = pc.b, kvh = pc.kvh, prior = pc.prior, nn = pc.nn, t0 = pc.t0, h0 = pc.h0, nh = pc.nh;
    const int kmax = pc.kmax, nkt_all = pc.nkt_all, kt0 = pc.kt0, nkt = pc.nkt;
    const int full_below = pc.full_below;                   // keys <= this are visible to every row
    const int unit_row0 = (b * p.Hkv + kvh) * p.max_len;    // first cache row of (b, kvh)
    // Window bounds of the block's rows: keys <= min_lo are outside every row's
    // window, keys > max_lo inside every row's window (-1: no window).
    const int min_lo = kWin ? full_below - p.window : -1;
    const int max_lo = kWin ? kmax - p.window : -1;
    auto slot_row = [&](int kt) {
        if (!p.pg.table) return unit_row0 + ((kWin && p.ring) ? (kt * 128) % p.max_len : kt * 128);
        bool bad = false;  // paged: the tile lies in one page
        const int row = phys_row(p.pg, 0, p.Hkv, p.max_len, b, kvh, kt * 128, &bad);
        if (bad) atomicExch(p.err, kDevBadPage);
        return row;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int qbar = kF8 ? kBarQRaw : kBarQ;
            ptx::mbar_arrive_expect_tx(bar(qbar), nh * kTile128);
            for (int i = 0; i < nh; ++i) {
                // mode 0: 128 positions of head h0 + i; modes 1, 2: 128 packed rows
                const int qrow = (p.mode == 0) ? ((b * p.Hq) + h0 + i) * p.T + t0
                                               : (b * p.Hq + h0) * p.T + pc.pr0 + i * 128;
                for (int hf = 0; hf < 2; ++hf)
                    ptx::tma_load_2d(sbase + kOffQ + i * kTile128 + hf * kBoxBytes, &tmQ, hf * 64, qrow, bar(qbar));
            }
            for (int j = 0; j < nkt && !*abort_flag; ++j) {
                const int s = j & 1;
                const int row = slot_row(kt0 + j);
                if (j >= 2 && !ptx::mbar_wait_bounded(bar(kBarKEmpty + s), ((j >> 1) & 1) ^ 1, kWaitNs)) {
                    atomicExch(p.err, kDevTimeoutEmpty);
                    *abort_flag = 1;
                    break;
                }
                if constexpr (kF8) {  // one 128 x 128-byte box into the stage's second half
                    ptx::mbar_arrive_expect_tx(bar(kBarKRaw + s), kBoxBytes);
                    ptx::tma_load_2d(sbase + kOffK + s * kTile128 + kBoxBytes, &tmK, 0, row, bar(kBarKRaw + s));
                } else {
                    ptx::mbar_arrive_expect_tx(bar(kBarKFull + s), kTile128);
                    for (int hf = 0; hf < 2; ++hf)
                        ptx::tma_load_2d(sbase + kOffK + s * kTile128 + hf * kBoxBytes, &tmK, hf * 64, row,
                                         bar(kBarKFull + s));
                }
                if (j >= 2 && !ptx::mbar_wait_bounded(bar(kBarVEmpty + s), ((j >> 1) & 1) ^ 1, kWaitNs)) {
                    atomicExch(p.err, kDevTimeoutEmpty);
                    *abort_flag = 1;
                    break;
                }
                if constexpr (kF8) {
                    ptx::mbar_arrive_expect_tx(bar(kBarVRaw + s), kBoxBytes);
                    ptx::tma_load_2d(sbase + kOffV + s * kTile128 + kBoxBytes, &tmV, 0, row, bar(kBarVRaw + s));
                } else {
                    ptx::mbar_arrive_expect_tx(bar(kBarVFull + s), kTile128);
                    for (int hf = 0; hf < 2; ++hf)
                        ptx::tma_load_2d(sbase + kOffV + s * kTile128 + hf * kBoxBytes, &tmV, hf * 64, row,
                                         bar(kBarVFull + s));
                }
            }
        }
    } else if (kF8 && (warp == 2 || warp == 3)) {
        // ------------------------------------------------------------ E4M3 -> f16 converters
        const int ct = tid - 64;
        auto wait_raw = [&](int b_idx, int parity) {
            if (!ptx::mbar_wait_bounded(bar(b_idx), parity, *abort_flag ? 0ull : kWaitNs)) {
                atomicExch(p.err, kDevTimeoutFull);
                *abort_flag = 1;
            }
        };
        auto ready = [&](int b_idx) {  // generic writes -> visible to the tensor core, then arrive
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(b_idx));
        };
        wait_raw(kBarQRaw, 0);
        convert_bf16_tiles(smem + kOffQ, nh * kTile128, ct);
        ready(kBarQ);
        for (int j = 0; j < nkt; ++j) {
            const int s = j & 1;
            wait_raw(kBarKRaw + s, (j >> 1) & 1);
            convert_e4m3_tile(smem + kOffK + s * kTile128, ct);
            ready(kBarKFull + s);
            wait_raw(kBarVRaw + s, (j >> 1) & 1);
            convert_e4m3_tile(smem + kOffV + s * kTile128, ct);
            ready(kBarVFull + s);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t id_qk = instr_desc(false, kF8), id_pv = instr_desc(true, kF8);
        auto wait = [&](int b_idx, int parity) {
            if (!ptx::mbar_wait_bounded(bar(b_idx), parity, *abort_flag ? 0ull : kWaitNs)) {
                atomicExch(p.err, kDevTimeoutFull);
                *abort_flag = 1;
            }
        };
        auto issue_s = [&](int i, int j, int qi) {  // S_i = Q_qi K_j^T
            const uint32_t qa = sbase + kOffQ + qi * kTile128, ka = sbase + kOffK + (j & 1) * kTile128;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * kBoxBytes + (k & 3) * 32;
                mma_ss(tmem + i * 128, smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024), id_qk, k > 0);
            }
            mma_commit(bar(kBarS + i));
        };
        auto issue_pv = [&](int i, int j, bool acc) {  // O_i (+)= P_i V_j (P_i in TMEM over S_i)
            const uint32_t va = sbase + kOffV + (j & 1) * kTile128;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_ts(tmem + 256 + i * 128, tmem + i * 128 + k * 8, smem_desc(va + k * 2048, kBoxBytes, 1024), id_pv,
                       (acc || k > 0) ? 1u : 0u);
            mma_commit(bar(kBarO + i));
        };
        // Mode 2 (one packed row tile): key tile j goes to S/O buffer j & 1,
        // which is also its K/V stage, so one buffer's softmax overlaps the
        // other's MMAs.  Issue order S(0), S(1), PV(0), S(2), PV(1), S(3), ...
        constexpr bool alt = kAlt;
        if (lane == 0) {
            wait(kBarQ, 0);
            wait(kBarKFull, 0);
            tc_fence_after();
            issue_s(0, 0, 0);
            if (!alt && nh == 2) issue_s(1, 0, 1);
            mma_commit(bar(kBarKEmpty + 0));
            if (alt && nkt > 1) {
                wait(kBarKFull + 1, 0);
                tc_fence_after();
                issue_s(1, 1, 0);
                mma_commit(bar(kBarKEmpty + 1));
            }
        }
        for (int j = 0; j < nkt; ++j) {
            const int s = j & 1;
            // V rows past the block's last visible key: clear them (whole warp)
            // before the PV MMAs read the stage.
            if (lane == 0) wait(kBarVFull + s, (j >> 1) & 1);
            __syncwarp();
            const int key0 = (kt0 + j) * 128;
            if (kt0 + j == nkt_all - 1 || (kWin && key0 <= min_lo)) {
                // rows [0, vr1) are outside every row's window, rows [vr0, 128)
                // past the last visible key
                const int vr0 = min(128, kmax - key0 + 1), vr1 = max(0, min(128, min_lo - key0 + 1));
                uint8_t* vb = smem + kOffV + s * kTile128;
                const int per_hi = (128 - vr0) * 8, per_lo = vr1 * 8;
#pragma unroll 1
                for (int idx = lane; idx < 2 * (per_hi + per_lo); idx += 32) {
                    const int hf = idx / (per_hi + per_lo), rem = idx - hf * (per_hi + per_lo);
                    const int row = rem < per_lo ? (rem >> 3) : vr0 + ((rem - per_lo) >> 3);
                    *reinterpret_cast<uint4*>(vb + hf * kBoxBytes + row * 128 + (rem & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0 && alt) {
                wait(kBarP + s, (j >> 1) & 1);
                tc_fence_after();
                issue_pv(s, j, j >= 2);
                mma_commit(bar(kBarVEmpty + s));
                if (j + 2 < nkt) {
                    wait(kBarKFull + s, ((j + 2) >> 1) & 1);
                    tc_fence_after();
                    issue_s(s, j + 2, 0);
                    mma_commit(bar(kBarKEmpty + s));
                }
            } else if (lane == 0) {
                wait(kBarP + 0, j & 1);
                tc_fence_after();
                issue_pv(0, j, j > 0);
                if (j + 1 < nkt) {
                    wait(kBarKFull + ((j + 1) & 1), ((j + 1) >> 1) & 1);
                    tc_fence_after();
                    issue_s(0, j + 1, 0);
                }
                if (nh == 2) {
                    wait(kBarP + 1, j & 1);
                    tc_fence_after();
                    issue_pv(1, j, j > 0);
                }
                mma_commit(bar(kBarVEmpty + s));
                if (j + 1 < nkt) {
                    if (nh == 2) issue_s(1, j + 1, 1);
                    mma_commit(bar(kBarKEmpty + ((j + 1) & 1)));
                }
            }
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax (one thread per query row)
        const int i = (warp - 4) >> 2;  // S/O buffer: row tile of the pair, or in mode 2 key-tile parity
        const int r = tid & 127;        // row in the block = TMEM lane
        constexpr bool alt = kAlt;
        if (i < nh || alt) {
            const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const uint32_t tS = tmem + lane_off + i * 128, tO = tmem + lane_off + 256 + i * 128;
            int lim;
            if (p.mode == 0) {
                const int t = t0 + r;
                lim = ((t < nn) && (t < p.T)) ? prior + t : -1;
            } else {
                const int pr = pc.pr0 + (alt ? 0 : i * 128) + r;  // packed row g*T + t of the KV head
                const int t = pr % p.T;
                lim = ((pr < p.G * p.T) && (t < nn)) ? prior + t : -1;
            }
            const bool valid = lim >= 0;
            // key tiles of this buffer: all of the piece's, or in mode 2 every other one
            const int jfirst = alt ? i : 0, jstep = alt ? 2 : 1;
            const int nloc = alt ? (nkt - i + 1) / 2 : nkt;
            const int lo_row = (kWin && valid) ? lim - p.window : -(1 << 30);  // keys <= lo_row: outside the window
            // score scale in base 2 (times the K scale of an FP8 cache)
            const float sl2 = kF8 ? p.scale_log2 * p.kscale[kvh] : p.scale_log2;
            float m_ref = -INFINITY, l = 0.f;
            for (int jj = 0; jj < nloc; ++jj) {
                const int j = jfirst + jj * jstep;
                if (!ptx::mbar_wait_bounded(bar(kBarS + i), jj & 1, *abort_flag ? 0ull : kWaitNs)) {
                    atomicExch(p.err, kDevTimeoutFull);
                    *abort_flag = 1;
                }
                tc_fence_after();
                const bool full_tile = ((kt0 + j) * 128 + 127 <= full_below) && (!kWin || (kt0 + j) * 128 > max_lo);
                const int key0 = (kt0 + j) * 128;
                // pass 1: row max of the raw scores (scale > 0, so it scales after);
                // 64 columns per TMEM load, one wait each.  The 64-column chunks of
                // both passes and of the rescale are not unrolled: each waits on its
                // own TMEM load anyway, and the smaller loop body keeps the kernel's
                // code and registers down (127 registers against 162 to 168
                // unrolled; the FP8 variant ran 17 % faster).
                float mx = -INFINITY;
                uint32_t v[64];
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    tmem_ld64(tS + c * 64, v);
                    tmem_ld_wait();
                    if (full_tile) {
#pragma unroll
                        for (int e = 0; e < 64; e += 2) mx = fmax3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
                    } else {
                        const int kl = lim - key0 - c * 64;    // elements e <= kl are visible
                        const int kll = kWin ? lo_row - key0 - c * 64 : -1;  // ... and e > kll (the window)
#pragma unroll
                        for (int e = 0; e < 64; ++e)
                            if (e <= kl && e > kll) mx = fmaxf(mx, __uint_as_float(v[e]));
                    }
                }
                mx = (mx == -INFINITY) ? -INFINITY : mx * sl2;
                const bool move = mx > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mx != -INFINITY);
                if (__any_sync(0xffffffffu, move)) {
                    // Move the reference max.  O_i holds the PV sums up to tile
                    // j-1 (all with the old reference): wait for the last of them
                    // and scale O_i and l by 2^(old - new).  The TMEM loads and
                    // stores are warp-collective, so the warp rescales together;
                    // rows that keep their reference scale by 1.
                    const float f = !move ? 1.f : (m_ref == -INFINITY) ? 0.f : ptx::ex2(m_ref - mx);
                    if (jj > 0) {
                        if (!ptx::mbar_wait_bounded(bar(kBarO + i), (jj - 1) & 1, *abort_flag ? 0ull : kWaitNs)) {
                            atomicExch(p.err, kDevTimeoutFull);
                            *abort_flag = 1;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < 2; ++c) {
                            tmem_ld64(tO + c * 64, v);
                            tmem_ld_wait();
                            uint32_t w[32];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(v[h * 32 + e]) * f);
                                tmem_st32(tO + c * 64 + h * 32, w);
                            }
                        }
                        tmem_st_wait();
                    }
                    l *= f;
                    if (move) m_ref = mx;
                }
                // pass 2: p = 2^(s * scale - m_ref) as bf16 pairs into TMEM over S_i
                const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
                const uint64_t sc2 = f2pack(sl2, sl2), nmu2 = f2pack(-mu, -mu);
                uint64_t sum2 = f2pack(0.f, 0.f);
                uint32_t pk[32];
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    tmem_ld64(tS + c * 64, v);
                    tmem_ld_wait();
                    const int kl = full_tile ? 1 << 30 : lim - key0 - c * 64;
                    const int kll = (full_tile || !kWin) ? -1 : lo_row - key0 - c * 64;
#pragma unroll
                    for (int e = 0; e < 64; e += 2) {
                        float x0, x1;
                        f2unpack(ffma2(f2pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2, nmu2), x0, x1);
                        float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        if (!full_tile) {
                            if (e > kl || e <= kll) p0 = 0.f;
                            if (e + 1 > kl || e + 1 <= kll) p1 = 0.f;
                        }
                        sum2 = fadd2(sum2, f2pack(p0, p1));
                        pk[e >> 1] = kF8 ? ptx::pack_f16x2(p0, p1) : ptx::pack_bf16x2(p0, p1);
                    }
                    // keys c*64 .. c*64+63 -> P columns c*32 .. c*32+31 (S columns already read)
                    tmem_st32(tS + c * 32, pk);
                }
                {
                    float s0, s1;
                    f2unpack(sum2, s0, s1);
                    l += s0 + s1;
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(kBarP + i));
            }
            // epilogue: O_i / l for valid rows
            if (nloc > 0 && !ptx::mbar_wait_bounded(bar(kBarO + i), (nloc - 1) & 1, *abort_flag ? 0ull : kWaitNs)) {
                atomicExch(p.err, kDevTimeoutFull);
                *abort_flag = 1;
            }
            tc_fence_after();
            if (alt) {
                // Merge the odd-tile state (m, l, O_1) into the even-tile one:
                // o = (2^(m0-M) O_0 + 2^(m1-M) O_1) / (2^(m0-M) l0 + 2^(m1-M) l1).
                // Both buffers sit in the same TMEM lanes, so warpgroup 0 reads
                // O_1 directly once warpgroup 1 has seen its last PV land.
                float* ml1 = reinterpret_cast<float*>(smem + kOffQ + kTile128);  // second Q tile: unused here
                if (i == 1) {
                    ml1[r] = m_ref;
                    ml1[128 + r] = l;
                }
                tc_fence_before();
                ptx::named_barrier_sync(3, 256);
                tc_fence_after();
                if (i == 0 && nkt > 1) {
                    const float m1 = ml1[r], l1 = ml1[128 + r];
                    const float M = fmaxf(m_ref, m1);
                    const float Mu = (M == -INFINITY) ? 0.f : M;
                    const float f0 = (m_ref == -INFINITY) ? 0.f : ptx::ex2(m_ref - Mu);
                    const float f1 = (m1 == -INFINITY) ? 0.f : ptx::ex2(m1 - Mu);
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t w0[32], w1[32];
                        tmem_ld32(tO + c * 32, w0);
                        tmem_ld32(tO + 128 + c * 32, w1);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            w0[e] = __float_as_uint(__uint_as_float(w0[e]) * f0 + __uint_as_float(w1[e]) * f1);
                        tmem_st32(tO + c * 32, w0);
                    }
                    tmem_st_wait();
                    m_ref = M;
                    l = l * f0 + l1 * f1;
                }
            }
            // output row: head h0 + i, position t0 + r (mode 0), or packed row pr of the KV head
            const int qrow = (p.mode == 0) ? ((b * p.Hq) + h0 + i) * p.T + t0 + r
                                           : (b * p.Hq + h0) * p.T + pc.pr0 + (alt ? 0 : i * 128) + r;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(qrow) * kD;
            if (alt && i == 1) {
                // state handed to warpgroup 0
            } else if (pc.slot != kPrefillNoSlot) {
                split_epilogue(p.partials, p.err, tS, tO, i, r, valid, m_ref, l, pc.slot, pc.kidx, pc.npc, dst, merge_flag,
                               kF8 ? p.vscale[kvh] : 1.f,
                               reinterpret_cast<float*>(smem + kOffQ + i * kSplitStageBytes));
            } else {
            const float inv = (valid && l > 0.f) ? (kF8 ? p.vscale[kvh] : 1.f) / l : 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[32];
                tmem_ld32(tO + c * 32, w);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 q4;
                        q4.x = ptx::pack_bf16x2(__uint_as_float(w[e]) * inv, __uint_as_float(w[e + 1]) * inv);
                        q4.y = ptx::pack_bf16x2(__uint_as_float(w[e + 2]) * inv, __uint_as_float(w[e + 3]) * inv);
                        q4.z = ptx::pack_bf16x2(__uint_as_float(w[e + 4]) * inv, __uint_as_float(w[e + 5]) * inv);
                        q4.w = ptx::pack_bf16x2(__uint_as_float(w[e + 6]) * inv, __uint_as_float(w[e + 7]) * inv);
                        *reinterpret_cast<uint4*>(dst + c * 32 + e) = q4;
                    }
                }
            }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

}  // namespace

size_t prefill_smem_bytes() { return kSmemPF; }

cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                              const CUtensorMap& tmV, cudaStream_t stream) {
    static bool attr_set = false;
    if (!attr_set) {
        for (auto* k : {prefill_tc_kernel<false, false, false>, prefill_tc_kernel<true, false, false>,
                        prefill_tc_kernel<false, true, false>, prefill_tc_kernel<true, true, false>,
                        prefill_tc_kernel<false, false, true>, prefill_tc_kernel<true, false, true>,
                        prefill_tc_kernel<false, true, true>, prefill_tc_kernel<true, true, true>}) {
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kSmemPF));
            if (e != cudaSuccess) return e;
        }
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_pieces);
    cfg.blockDim = dim3(kThreadsPF);
    cfg.dynamicSmemBytes = kSmemPF;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool win = p.window > 0 || p.ring;
    const bool alt = p.mode == 2;
    using Kernel = void (*)(PrefillParams, CUtensorMap, CUtensorMap, CUtensorMap);
    Kernel k;
    if (p.fp8)
        k = win ? (alt ? prefill_tc_kernel<true, true, true> : prefill_tc_kernel<true, false, true>)
                : (alt ? prefill_tc_kernel<false, true, true> : prefill_tc_kernel<false, false, true>);
    else
        k = win ? (alt ? prefill_tc_kernel<true, true, false> : prefill_tc_kernel<true, false, false>)
                : (alt ? prefill_tc_kernel<false, true, false> : prefill_tc_kernel<false, false, false>);
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, p, tmQ, tmK, tmV);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kvc
