// Device-side helpers shared by the CUDA translation units: pool addressing, 16-bit
// conversions and the per-translation-unit copy of the format constants.
#pragma once

#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include "kvq_internal.h"

namespace kvq {

// Each translation unit holds its own copy (no relocatable device code); the host
// uploads the same values to every copy once.
static __constant__ FormatTables c_tab;

__device__ __forceinline__ char* pool_at(const void* pool, int64_t off) {
    return (char*)pool + off;
}

__device__ __forceinline__ uint16_t* sink_row(const Layout& L, const void* pool, int w, int64_t unit, int pos) {
    return (uint16_t*)pool_at(pool, L.sink_off[w] + unit * L.sink_stride[w]) + (int64_t)pos * L.D;
}
// tq6_0 journal: code row (D/128 blocks of [ql 64 | qh 32]) and scale row (D/128 fp16).
__device__ __forceinline__ uint8_t* jcode_row(const Layout& L, const void* pool, int w, int64_t unit, int slot) {
    return (uint8_t*)pool_at(pool, L.jcode_off[w] + unit * L.jcode_stride[w]) + (int64_t)slot * L.jrow_bytes;
}
__device__ __forceinline__ uint16_t* jscale_row(const Layout& L, const void* pool, int w, int64_t unit, int slot) {
    return (uint16_t*)pool_at(pool, L.jscale_off[w] + unit * L.jscale_stride[w]) + (int64_t)slot * (L.D / 128);
}
// Exact journal row (16-bit, D values) shares the jcode area.
__device__ __forceinline__ uint16_t* jexact_row(const Layout& L, const void* pool, int w, int64_t unit, int slot) {
    return (uint16_t*)pool_at(pool, L.jcode_off[w] + unit * L.jcode_stride[w]) + (int64_t)slot * L.D;
}
__device__ __forceinline__ uint16_t* tail_row(const Layout& L, const void* pool, int w, int64_t unit, int slot) {
    return (uint16_t*)pool_at(pool, L.tail_off[w] + unit * L.tail_stride[w]) + (int64_t)slot * L.D;
}
__device__ __forceinline__ uint8_t* body_rec(const Layout& L, const void* pool, int w, int64_t unit, int g) {
    return (uint8_t*)pool_at(pool, L.body_off[w] + unit * L.body_stride[w]) + (int64_t)g * L.rec_bytes[w];
}
__device__ __forceinline__ uint32_t* status_word(const Layout& L, const void* pool) {
    return (uint32_t*)pool_at(pool, L.status_off);
}

__device__ __forceinline__ int journal_slot(const Layout& L, int pos) { return (pos - kSink) % L.R; }

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ float x16_to_f(uint16_t b, int fmt) { return fmt == KVQ_BF16 ? bf2f(b) : h2f(b); }
__device__ __forceinline__ uint16_t f2h_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint16_t f2bf_bits(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// -1 where bit i of the splitmix64 sign words is set (i < 128; set 0 = s1, 1 = s2).
__device__ __forceinline__ bool sign_neg(int set, int i) {
    return (c_tab.sign_words[2 * set + (i >> 6)] >> (i & 63)) & 1ULL;
}

// One sealed group of a seal launch: group index gidx counts the layers' groups in order,
// the sequences of the batch in order inside a layer.
struct SealTaskPos { int layer, slot, g, pos0, b; };   // b: index in the launch's sequence list

__device__ __forceinline__ SealTaskPos seal_task(const SealParams& p, int gidx) {
    SealTaskPos t;
    t.layer = p.layer0 + gidx / p.groups_per_layer;
    const int r = gidx % p.groups_per_layer;
    int b = 0;
    while (b + 1 < p.n_seq && p.seq[b + 1].prefix <= r) ++b;
    const int gi = r - p.seq[b].prefix;
    t.slot = p.seq[b].slot;
    t.g = p.seq[b].first_group + gi;
    t.pos0 = p.seq[b].first_pos + kGroup * gi;
    t.b = b;
    return t;
}

__device__ __forceinline__ void flag_nonfinite(const Layout& L, const void* pool, float x) {
    if (!isfinite(x)) atomicOr(status_word(L, pool), 1u);
}

// Programmatic dependent launch (sm_90 and later). A kernel launched with programmatic stream
// serialization may be scheduled before the launch ahead of it in the stream has finished:
// as that launch's CTAs exit, or once every one of them has executed grid_dep_launch.
// grid_dep_wait blocks until the launches it depends on have completed and their memory
// operations are visible; it returns at once in a kernel launched without the attribute.
// Every kernel launched this way executes grid_dep_wait before its first global memory access,
// except the decode kernel's items when the launch ahead is the merge kernel (AttnParams::early).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets the next launch in the stream start. Only the merge kernel calls it, after its own
// grid_dep_wait: when the next launch starts, the launch ahead of the merge has completed.
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Launches kernel k; with pdl, with programmatic stream serialization (see above).
template <typename... P, typename... A>
inline cudaError_t launch_k(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                            A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, std::forward<A>(args)...);
}

}  // namespace kvq
