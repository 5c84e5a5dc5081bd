// Device helpers shared by the streaming decode kernels (body records and region rows):
// mbarrier / cp.async.bulk wrappers with bounded waits, the consumer-warp named barrier,
// mma.sync m16n8k16, exact fp16 code decoders, and the query / output rotations.
#pragma once
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cfloat>
#include "device_common.cuh"

namespace kvq {
namespace {


constexpr int kConsumers = 8;
constexpr int kCT = kConsumers * 32;                 // consumer threads
constexpr int kBodyThreads = kCT + 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTbqScale = 0.0883883461356163f;
constexpr int kLutBytes = 256 * 32 * 4;
constexpr uint64_t kWaitNs = 2000000000ull;          // bounded waits: 2 s, then the status word is set

// fragment decoder families of the streaming decode kernel: KVarN codes, TBQ4 centroid pairs,
// Q8_0 / Q4_0 blocks, and (keys only) Q5_1 (min-offset 5-bit blocks of 32) and tq5_0 (rotated
// symmetric 5-bit blocks of 128)
enum { KF_KVARN = 0, KF_TBQ4 = 1, KF_Q8 = 2, KF_Q4 = 3, KF_Q51 = 4, KF_TQ5 = 5 };

// ------------------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t gtime() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }\n"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait on an mbarrier phase (limit_ns of %globaltimer). On timeout it sets bit 1 of
// the status word and the CTA's abort flag; once the flag is set no thread waits again (the
// CTA runs to its end on stale data, reaching every barrier, and the host learns of it from
// the status word).
__device__ __forceinline__ bool mbar_wait_ns(uint32_t bar, uint32_t parity, uint32_t* status, volatile int* abort_flag,
                                             uint64_t limit_ns) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtime();
    while (!mbar_try(bar, parity)) {
        if (*abort_flag) return false;
        if (gtime() - t0 > limit_ns) {
            atomicOr(status, 2u);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status, volatile int* abort_flag) {
    return mbar_wait_ns(bar, parity, status, abort_flag, kWaitNs);
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kCT) : "memory"); }
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------------------ code decode
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t as_u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ uint32_t pack_f2(float a, float b) { return as_u(__floats2half2_rn(a, b)); }
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) { return as_u(__hmul2(as_h2(a), as_h2(b))); }
// Nibbles x and x+4 of w (x = 0..3) as half2 (64 + n_x, 64 + n_x+4), exact: each nibble moved
// to mantissa bits 4-7 of a half with exponent 6.
__device__ __forceinline__ uint32_t nib64(uint32_t w, int x) {
    const uint32_t t = (x == 0) ? (w << 4) : (w >> (4 * x - 4));
    return (t & 0x00F000F0u) | 0x54005400u;
}
// Adds 16 x bit x (low half) and 16 x bit x+4 (high half) of h to a nib64 pair: mantissa bit 8.
__device__ __forceinline__ uint32_t add_bit5(uint32_t raw, uint32_t h, int x) {
    const uint32_t t = ((h >> x) & 0x11u) * 0x00100100u;
    return (t & 0x01000100u) | raw;
}
// Signed bytes of w (sel 0x5140: bytes 0,1; 0x7362: bytes 2,3) as half2 (1152 + b), exact.
__device__ __forceinline__ uint32_t i8raw(uint32_t w, uint32_t sel) {
    return __byte_perm(w ^ 0x80808080u, 0x64646464u, sel);
}
__device__ __forceinline__ uint32_t movtrans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
    return d;
}
__device__ __forceinline__ float lo_f(uint32_t u) { return __low2float(as_h2(u)); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __high2float(as_h2(u)); }

// Forward rotation of one block (n = 32 NK values, value i = lane + 32 k in v[k]) of a query
// row with warp shuffles: FWHT butterflies, strides ascending, then scale and signs.
template <int NK>
__device__ __forceinline__ void warp_rotate(float (&v)[NK], int lane, int rot) {
    if (rot == ROT_NONE) return;
    if (rot == ROT_TBQ128) {
#pragma unroll
        for (int k = 0; k < NK; ++k)
            if (sign_neg(0, lane + 32 * k)) v[k] = -v[k];
    }
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const bool upper = lane & s;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const float o = __shfl_xor_sync(0xffffffffu, v[k], s);
            v[k] = upper ? (o - v[k]) : (v[k] + o);
        }
    }
#pragma unroll
    for (int m = 1; m < NK; m <<= 1)
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            if (k & m) continue;
            const float a = v[k], c = v[k + m];
            v[k] = a + c;
            v[k + m] = a - c;
        }
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        if (rot == ROT_HAD256) v[k] *= 0.0625f;
        else if (rot == ROT_TBQ128) v[k] = (sign_neg(1, lane + 32 * k) ? -v[k] : v[k]) * kTbqScale;
    }
}

// Inverse rotation of one block (n = 32 NK values, value i = lane + 32 k in v[k]) with warp
// shuffles: HAD256: FWHT x 1/16; TBQ128: second sign set, FWHT, first sign set x scale.
template <int NK>
__device__ __forceinline__ void warp_unrotate(float (&v)[NK], int lane, int rot) {
    if (rot == ROT_NONE) return;
    if (rot == ROT_TBQ128) {
#pragma unroll
        for (int k = 0; k < NK; ++k)
            if (sign_neg(1, lane + 32 * k)) v[k] = -v[k];
    }
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const bool upper = lane & s;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const float o = __shfl_xor_sync(0xffffffffu, v[k], s);
            v[k] = upper ? (o - v[k]) : (v[k] + o);
        }
    }
#pragma unroll
    for (int m = 1; m < NK; m <<= 1)
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            if (k & m) continue;
            const float a = v[k], c = v[k + m];
            v[k] = a + c;
            v[k + m] = a - c;
        }
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        if (rot == ROT_HAD256) v[k] *= 0.0625f;
        else v[k] = (sign_neg(0, lane + 32 * k) ? -v[k] : v[k]) * kTbqScale;
    }
}

// Writes a work item's partial: m and l per query row, then o (rows [NQ][D] in shared memory,
// fp32) rotated back to the original domain by warp shuffles (one warp per row block) and
// stored straight to global memory. Called by the consumer threads after a consumer barrier.
template <int D, int NQ>
__device__ __forceinline__ void write_partial(const float* ofin, const float* m, const float* l, float* part,
                                              int rot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < NQ) {
        part[threadIdx.x] = m[threadIdx.x];
        part[NQ + threadIdx.x] = l[threadIdx.x];
    }
    float* po = part + 2 * NQ;
    if (rot == ROT_HAD256) {
        if constexpr (D >= 256) {
            for (int u = warp; u < NQ * (D / 256); u += kConsumers) {
                const int base = (u / (D / 256)) * D + (u % (D / 256)) * 256;
                float v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = ofin[base + lane + 32 * k];
                warp_unrotate<8>(v, lane, rot);
#pragma unroll
                for (int k = 0; k < 8; ++k) po[base + lane + 32 * k] = v[k];
            }
        }
    } else {
        for (int u = warp; u < NQ * (D / 128); u += kConsumers) {
            const int base = (u / (D / 128)) * D + (u % (D / 128)) * 128;
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = ofin[base + lane + 32 * k];
            warp_unrotate<4>(v, lane, rot);
#pragma unroll
            for (int k = 0; k < 4; ++k) po[base + lane + 32 * k] = v[k];
        }
    }
}

// Consumer-wide FWHT over rows of n values (fp32 shared memory), for the inverse rotation.
__device__ void fwht_rows_c(float* xs, int total, int n) {
    for (int s = 1; s < n; s <<= 1) {
        for (int p = threadIdx.x; p < total / 2; p += kCT) {
            const int blk = p / (n / 2), q = p % (n / 2);
            const int i = blk * n + (q / s) * 2 * s + (q % s);
            const float a = xs[i], c = xs[i + s];
            xs[i] = a + c;
            xs[i + s] = a - c;
        }
        csync();
    }
}
__device__ void inverse_rotate_c(float* xs, int rows, int D, int rot) {
    const int total = rows * D;
    if (rot == ROT_HAD256) {
        fwht_rows_c(xs, total, 256);
        for (int i = threadIdx.x; i < total; i += kCT) xs[i] *= 0.0625f;
        csync();
    } else if (rot == ROT_TBQ128) {
        for (int i = threadIdx.x; i < total; i += kCT)
            if (sign_neg(1, i & 127)) xs[i] = -xs[i];
        csync();
        fwht_rows_c(xs, total, 128);
        for (int i = threadIdx.x; i < total; i += kCT) {
            float y = xs[i];
            if (sign_neg(0, i & 127)) y = -y;
            xs[i] = y * kTbqScale;
        }
        csync();
    }
}

}  // namespace
}  // namespace kvq
