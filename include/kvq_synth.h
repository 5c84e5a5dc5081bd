/*
 * kvq_synth.h — seeded synthetic fp16 inputs on the device, for tests and benchmarks.
 *
 * Not a step of the KV-cache method: it fills buffers with the same values the Python
 * generator (quantized_kv_cache_gb300/synth.py) draws on the host, bit for bit, so large
 * workloads can be built in HBM without host copies. Element i of stream `key` is
 * NORMAL_TABLE[mix64(key + (i + 1) * 0x9E3779B97F4A7C15) >> 48], with mix64 the splitmix64
 * output function (Steele, Lea & Flood 2014) and NORMAL_TABLE a caller-supplied device
 * table of 65,536 fp16 values.
 */
#ifndef KVQ_SYNTH_H
#define KVQ_SYNTH_H

#include <stdint.h>
#include "kvq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* kvq_synth_fill — out: device fp16 [n_pos][n_heads][head_dim].
 * Element (p, h, c) = fp16(fp32(v) * factor[h][c]) with v element (pos0 + p) * head_dim + c
 * of the stream head_keys[h]; factor is a device fp32 [n_heads][head_dim] array, or NULL
 * for factor 1 (v verbatim). head_keys: host uint64 [n_heads]. table: device fp16 [65536].
 * KVQ_EINVAL on null / misaligned pointers or non-positive sizes. */
kvq_status kvq_synth_fill(void* out, int64_t n_pos, int n_heads, int head_dim,
                          const uint64_t* head_keys, int64_t pos0, const float* factor,
                          const void* table, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_SYNTH_H */
