// Append of one position of one (layer, sequence, KV head, K or V): the exact copies and the
// rotated tq6_0 ring row. Shared by the append kernel and the fused decode step (whose region
// item that holds the newest position appends it).
//
// Every floating-point step uses the explicit round-to-nearest intrinsics, so no multiply-add
// is contracted whatever the unit's -fmad setting and the ring rows are reproducible bit for
// bit: one IEEE fp32 rounding per operation, round-half-even rint and fp16 casts.
#pragma once
#include <cuda_runtime.h>
#include "device_common.cuh"

namespace kvq {
namespace {
namespace codec {

constexpr float kTbqScale = 0.0883883461356163f;   // fp32(1/sqrt(128)) = 0x3DB504F3
constexpr float kHad256Scale = 0.0625f;             // 1/16, exact
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fdiv(float a, float b) { return __fdiv_rn(a, b); }
// Two of the same operations in one instruction (sm_100 and later): each half rounds to nearest
// on its own, so the results are those of fmul / fadd / __fmaf_rn bit for bit (checked
// elementwise on GB300). The code generator may contract a packed multiply whose result feeds
// a packed add into a packed multiply-add, explicit rounding modifiers notwithstanding (one
// row's sum of squares in eleven then differed): so no fmul2 result reaches an fadd2 or fsub2.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) { return __fadd2_rn(a, make_float2(-b.x, -b.y)); }
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float warp_max(float v) {
    for (int s = 16; s >= 1; s >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, s));
    return v;
}

// In-warp FWHT of a block of 32 * NK values, value index i = lane + 32 k held in v[k].
template <int NK>
__device__ __forceinline__ void warp_fwht(float (&v)[NK], int lane) {
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const bool upper = lane & s;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const float p = __shfl_xor_sync(kFull, v[k], s);
            v[k] = upper ? fsub(p, v[k]) : fadd(v[k], p);
        }
    }
#pragma unroll
    for (int m = 1; m < NK; m <<= 1) {
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            if (k & m) continue;
            const float a = v[k], b = v[k + m];
            v[k] = fadd(a, b);
            v[k + m] = fsub(a, b);
        }
    }
}

// One tq6_0 block (values lane + 32 m, m = 0..3, taken from v[k0 + m]) of a journal slot:
// scale, codes through shared memory, then the ql / qh planes.
template <int NK>
__device__ __forceinline__ void tq6_block(const float (&v)[NK], int k0, int blk, int lane, uint8_t* cs, uint8_t* row,
                                          uint16_t* sc) {
    float a = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) a = fmaxf(a, fabsf(v[k0 + m]));
    a = warp_max(a);
    const uint16_t d16 = f2h_bits(fdiv(a, 31.0f));
    const float d = h2f(d16);
    const float inv = (d == 0.f) ? 0.f : fdiv(1.0f, d);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        float q = (d == 0.f) ? 0.f : rintf(fmul(v[k0 + m], inv));
        q = fminf(fmaxf(q, -31.f), 31.f);
        cs[128 * blk + lane + 32 * m] = (uint8_t)((int)q + 32);
    }
    __syncwarp();
    const uint8_t* c = cs + 128 * blk;
    uint8_t* out = row + 96 * blk;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int j = lane + 32 * r;
        out[j] = (uint8_t)((c[2 * j] & 15) | ((c[2 * j + 1] & 15) << 4));
    }
    out[64 + lane] = (uint8_t)((c[4 * lane] >> 4) | ((c[4 * lane + 1] >> 4) << 2) | ((c[4 * lane + 2] >> 4) << 4) |
                               ((c[4 * lane + 3] >> 4) << 6));
    if (lane == 0) sc[blk] = d16;
}

// Appends the fp16 row src (D values) of one (layer, sequence slot, KV head) unit, w = 0 for K
// and 1 for V, at position pos: below position 128 the sink row; with an exact journal its
// slot (pos - 128) mod R; with the tq6_0 journal the exact tail slot pos mod T (when
// write_tail) and the rotated tq6_0 codes and block scales of ring slot (pos - 128) mod R.
// Threads [0, nthr) of the calling block take part (tid: this thread's index among them; nthr
// a multiple of 32, at least one warp per rotation block: D / 256 for HAD256, else D / 128);
// cs: D bytes of shared memory for the codes.
__device__ __forceinline__ void append_row(const Layout& L, const void* pool, int64_t unit, int w, int pos,
                                           const uint16_t* src, bool write_tail, int tid, int nthr, uint8_t* cs) {
    const int D = L.D;
    if (pos < kSink) {
        uint16_t* dst = sink_row(L, pool, w, unit, pos);
        for (int i = tid; i < D; i += nthr) dst[i] = src[i];
        return;
    }
    const int slot = journal_slot(L, pos);
    if (L.journal != KVQ_TQ6_0) {
        uint16_t* dst = jexact_row(L, pool, w, unit, slot);
        for (int i = tid; i < D; i += nthr) dst[i] = (L.journal == KVQ_BF16) ? f2bf_bits(h2f(src[i])) : src[i];
        return;
    }
    if (write_tail) {
        uint16_t* tl = tail_row(L, pool, w, unit, pos % L.T);
        for (int i = tid; i < D; i += nthr) tl[i] = (L.tail_fmt == KVQ_BF16) ? f2bf_bits(h2f(src[i])) : src[i];
    }
    // rotation: one warp per rotation block (256 values for HAD256, else 128), value
    // i = lane + 32 k of the block in v[k]; the butterflies, signs and scale are those of the
    // block-wide rotation, in the same order
    const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
    uint8_t* row = jcode_row(L, pool, w, unit, slot);
    uint16_t* sc = jscale_row(L, pool, w, unit, slot);
    if (L.rot == ROT_HAD256) {
        for (int u = warp; u < D / 256; u += nw) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = h2f(src[256 * u + lane + 32 * k]);
            warp_fwht<8>(v, lane);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = fmul(v[k], kHad256Scale);
            tq6_block(v, 0, 2 * u, lane, cs, row, sc);
            tq6_block(v, 4, 2 * u + 1, lane, cs, row, sc);
        }
    } else {
        for (int u = warp; u < D / 128; u += nw) {
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = h2f(src[128 * u + lane + 32 * k]);
            if (L.rot == ROT_TBQ128) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (sign_neg(0, lane + 32 * k)) v[k] = -v[k];
                warp_fwht<4>(v, lane);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float y = v[k];
                    if (sign_neg(1, lane + 32 * k)) y = -y;
                    v[k] = fmul(y, kTbqScale);
                }
            }
            tq6_block(v, 0, u, lane, cs, row, sc);
        }
    }
}

}  // namespace codec
}  // namespace
}  // namespace kvq
