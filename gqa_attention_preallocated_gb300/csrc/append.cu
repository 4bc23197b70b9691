// In-place KV append ("Implement grouped-query attention over a preallocated
// KV cache...", section "A strong answer", KVCache.append): row b's chunk
// k_new[b, h, 0:n_new[b], :] lands at K[b, h, lens[b] : lens[b]+n_new[b], :].
//
// For one (b, h) both the source rows and the destination rows are
// contiguous, so the copy is n_new[b] * d * elem bytes of 16-byte vectors:
// every thread moves one uint4, consecutive threads consecutive vectors, so
// loads and stores are fully coalesced 128-bit accesses.  blockIdx.y selects
// (h, K or V), blockIdx.z the row b.  In a ring cache ("Write the causal mask
// for a decode step...", "A strong answer": a ring buffer whose physical index
// is not the position) position a goes to slot a mod max_len.
//
// FP8 E4M3 caches ("16. Prefill, decode and the KV cache", exercise 4): the
// bf16 rows are quantized on the way in, each value x of KV head h stored as
// the E4M3 code of x * (1/scale[h]) (float32 reciprocal and product, round to
// nearest even, saturating at +-448); a thread turns one 16-byte source
// vector (8 values) into 8 bytes.

#include <cuda_bf16.h>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const __grid_constant__ AppendParams p) {
    // Chained launch: wait for the previous kernel in the stream to finish
    // (it may still read the cache or write the inputs), then let the next
    // kernel start its prologue.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int b = blockIdx.z;
    const int h = blockIdx.y >> 1;
    const bool is_v = (blockIdx.y & 1) != 0;
    const int n = p.n_new[b];
    const size_t bytes = static_cast<size_t>(n) * p.row_bytes;
    const size_t vec = static_cast<size_t>(blockIdx.x) * kAppendThreads + threadIdx.x;
    if (vec * 16 >= bytes) return;
    const size_t unit = static_cast<size_t>(b) * p.Hkv + h;
    const uint8_t* src = (is_v ? p.v_new : p.k_new) + unit * p.T * p.row_bytes;
    const uint4 val = __ldg(reinterpret_cast<const uint4*>(src) + vec);
    uint8_t* cache = is_v ? p.v_cache : p.k_cache;
    if (p.fp8) {
        const float inv = __frcp_rn(is_v ? p.vscale[h] : p.kscale[h]);
        const uint32_t w[4] = {val.x, val.y, val.z, val.w};
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)  // bf16 pair -> float32 (exact) -> scaled -> two E4M3 bytes
            c[i] = ptx::f32x2_to_e4m3x2(__fmul_rn(__uint_as_float(w[i] << 16), inv),
                                        __fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), inv));
        const uint2 q8 = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        const int dst_row = p.row_bytes / 2;  // d bytes a cache row
        const size_t byte = vec * 16, t = byte / p.row_bytes, off = (byte - t * p.row_bytes) / 2;
        bool bad = false;
        const int row = phys_row(p.pg, p.ring, p.Hkv, p.max_len, b, h, p.lens[b] + static_cast<int>(t), &bad);
        if (!bad) *reinterpret_cast<uint2*>(cache + static_cast<size_t>(row) * dst_row + off) = q8;
        return;
    }
    if (!p.ring && !p.pg.table) {
        uint8_t* base = cache + unit * p.max_len * p.row_bytes;
        reinterpret_cast<uint4*>(base + static_cast<size_t>(p.lens[b]) * p.row_bytes)[vec] = val;
    } else {
        // Ring or paged storage: the row of each position on its own.  A
        // position whose block-table entry is bad is not written (the next
        // attention call over it reports the entry).
        const size_t byte = vec * 16, t = byte / p.row_bytes;
        bool bad = false;
        const int row = phys_row(p.pg, p.ring, p.Hkv, p.max_len, b, h, p.lens[b] + static_cast<int>(t), &bad);
        if (!bad) *reinterpret_cast<uint4*>(cache + static_cast<size_t>(row) * p.row_bytes + (byte - t * p.row_bytes)) = val;
    }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int max_n_new, cudaStream_t stream) {
    const size_t vecs = (static_cast<size_t>(max_n_new) * p.row_bytes) / 16;
    dim3 grid(static_cast<unsigned>((vecs + kAppendThreads - 1) / kAppendThreads), 2u * p.Hkv, p.B);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kAppendThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kv_append_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kvc
