// Seeded synthetic fp16 inputs on the device (tests and benchmarks; not a step of the
// KV-cache method). Element i of the stream with key `key` is
// table[mix64(key + (i + 1) * 0x9E3779B97F4A7C15) >> 48], mix64 being the splitmix64 output
// function (Steele, Lea & Flood 2014); an optional per-(head, channel) fp32 factor scales
// the value before rounding back to fp16.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstdint>
#include "../../include/kvq_synth.h"
#include "kvq_internal.h"

namespace {

constexpr int kMaxHeads = 64;

struct SynthKeys {
    uint64_t key[kMaxHeads];
};

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__global__ void synth_kernel(uint16_t* out, int64_t n_pos, int n_heads, int head_dim, SynthKeys keys,
                             int64_t pos0, const float* factor, const uint16_t* table) {
    const int64_t total = n_pos * n_heads * head_dim;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(e % head_dim);
        const int h = (int)((e / head_dim) % n_heads);
        const int64_t p = e / ((int64_t)head_dim * n_heads);
        const uint64_t i = (uint64_t)(pos0 + p) * (uint64_t)head_dim + (uint64_t)c;
        const uint64_t z = mix64(keys.key[h] + (i + 1ULL) * 0x9E3779B97F4A7C15ULL);
        uint16_t v = table[z >> 48];
        if (factor) {
            const float f = factor[h * head_dim + c];
            v = __half_as_ushort(__float2half_rn(__fmul_rn(__half2float(__ushort_as_half(v)), f)));
        }
        out[e] = v;
    }
}

}  // namespace

extern "C" kvq_status kvq_synth_fill(void* out, int64_t n_pos, int n_heads, int head_dim,
                                     const uint64_t* head_keys, int64_t pos0, const float* factor,
                                     const void* table, void* stream) {
    if (!out || !head_keys || !table || n_pos <= 0 || n_heads <= 0 || n_heads > kMaxHeads || head_dim <= 0 ||
        pos0 < 0 || ((uintptr_t)out & 1) || ((uintptr_t)table & 1))
        return KVQ_EINVAL;
    SynthKeys k{};
    for (int h = 0; h < n_heads; ++h) k.key[h] = head_keys[h];
    const int64_t total = n_pos * n_heads * head_dim;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    synth_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>((uint16_t*)out, n_pos, n_heads, head_dim, k, pos0,
                                                                    factor, (const uint16_t*)table);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}
