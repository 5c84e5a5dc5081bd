// Seal of the scalar body formats (TBQ4, Q8_0, Q4_0): a persistent kernel in which every
// thread encodes one position of a 128-position group (SJ-KVaRN §2.1 item 4: full groups
// leave the journal as compact body records).
//
// Work unit ("tile"): one group x one KV head x K or V x one 128-channel block. The tile's
// 128 journal rows are staged in shared memory with 16-byte cp.async copies issued by all
// threads, rows padded to an odd multiple of 16 bytes so that the thread-per-row 16-byte
// reads are free of bank conflicts, three stages deep (two tiles in flight while one is
// encoded). Thread t decodes row t into 128 fp32 registers (tq6_0 codes spread a word at a
// time; 16-bit rows widened and, for TBQ4, rotated by an in-register FWHT), encodes it and
// writes its codes straight to the record: K (token-major) with 16-byte stores, V
// (channel-major) after a lane-shuffle transpose of 8 x 8 nibbles (4-bit codes) or 4 x 4
// bytes (Q8_0).
//
// Arithmetic is the codec's (tq6_0: SJ-KVaRN §2.1; TBQ4, Q8_0, Q4_0: KV cache math, table,
// "Worked example" and "rotate first"; HAL #582 §1): one IEEE fp32 rounding per operation
// through the _rn intrinsics (the unit is also built with -fmad=false), halving-tree sums,
// round-half-even. The TBQ4 index, the number of boundaries beta_k with u > beta_k, is read
// from a 2,048-bucket table indexed by the top 11 bits of an order-preserving integer key of u
// (sign, exponent, two mantissa bits): a bucket spans a value ratio of at most 1.25 and the
// boundaries of the 16-level Lloyd-Max table differ by a ratio of at least 1.28, so a bucket
// holds at most one boundary and idx = base[bucket] + (u > thr[bucket]), the same fp32
// comparison, taken on the keys as the carry of one 32-bit addition.
#include <cuda_runtime.h>
#include <algorithm>
#include "append_row.cuh"

namespace kvq {
namespace {

using namespace codec;

constexpr int kRows = 128;          // positions of a group = threads of a CTA
constexpr int kStages = 3;          // staged tiles per CTA
constexpr int kTq6Stride = 112;     // 96-byte tq6_0 block row + 16 bytes of padding
constexpr int kX16Stride = 272;     // 256-byte row of 128 16-bit values + 16 bytes of padding
constexpr int kBuckets = 2048;      // TBQ4 decision buckets (top 11 bits of an fp32 value)

// Row sources: the journal (tq6_0, F16 or BF16 rows), or the caller's fp16 input rows of a
// prefill chunk (J_IN: the values the journal would have held are formed from them on the way).
enum JournalKind { J_TQ6 = 0, J_F16 = 1, J_BF16 = 2, J_IN = 3 };

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// A tile's addresses, decoded once by thread 0 into a shared slot (the runtime divisions
// stay out of the other threads' path): rows = its first journal row (block offset
// included), scales = the tq6_0 scale rows, rec = the body record.
struct TileSlot {
    const uint8_t* rows;
    const uint8_t* scales;
    uint8_t* rec;
    int64_t rs;     // bytes from one position's 16-bit row to the next (16-bit sources)
    int w, b;
};
constexpr int kSlots = 64;       // ring of decoded tiles (iteration k in slot k % kSlots)
constexpr int kSlotBatch = 32;   // slots decoded together, by threads 4j (8 lanes in each warp)

// tile = ((group * H + head) * 2 + w) * (D / 128) + block
__device__ __forceinline__ TileSlot tile_slot(const Layout& L, const SealParams& p, int tile) {
    const int nb = L.D / 128;
    TileSlot t;
    t.b = tile % nb;
    int r = tile / nb;
    t.w = r & 1;
    r >>= 1;
    const int h = r % L.H;
    const SealTaskPos tk = seal_task(p, r / L.H);
    const int64_t unit = L.unit(tk.layer, tk.slot, h);
    const int s0 = journal_slot(L, tk.pos0);   // a group's 128 slots are contiguous
    t.rs = 2LL * L.D;
    if (p.k_src != nullptr) {
        const int64_t row = p.seq[tk.b].src_row + (tk.pos0 - p.seq[tk.b].first_pos);
        t.rows = reinterpret_cast<const uint8_t*>((t.w ? p.v_src : p.k_src) + (row * L.H + h) * L.D) + 256 * t.b;
        t.scales = nullptr;
        t.rs = 2LL * L.H * L.D;
    } else if (L.journal == KVQ_TQ6_0) {
        t.rows = jcode_row(L, p.pool, t.w, unit, s0) + 96 * t.b;
        t.scales = reinterpret_cast<const uint8_t*>(jscale_row(L, p.pool, t.w, unit, s0));
    } else {
        t.rows = reinterpret_cast<const uint8_t*>(jexact_row(L, p.pool, t.w, unit, s0)) + 256 * t.b;
        t.scales = nullptr;
    }
    t.rec = body_rec(L, p.pool, t.w, unit, tk.g);
    return t;
}

// Issues a tile's 128 journal rows (its 128-channel block) into a stage.
template <int JK>
__device__ __forceinline__ void issue_tile(const Layout& L, const TileSlot& t, uint8_t* st) {
    const int tid = threadIdx.x;
    if constexpr (JK == J_TQ6) {
        const int64_t jr = L.jrow_bytes;
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            const int c = tid + kRows * i, r = c / 6, k = c - 6 * r;
            cp_async16(st + r * kTq6Stride + 16 * k, t.rows + r * jr + 16 * k);
        }
        // the 128 rows' scales of every block ([128][D/128] fp16, 2D bytes)
        for (int c = tid; c < L.D / 8; c += kRows) cp_async16(st + kRows * kTq6Stride + 16 * c, t.scales + 16 * c);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = (tid >> 4) + 8 * i, k = tid & 15;
            cp_async16(st + r * kX16Stride + 16 * k, t.rows + r * t.rs + 16 * k);
        }
    }
}

// The tq6_0 staging of one 128-value block, in place: d = fp16(max|y| / 31), q = clamp(rint(y x
// (1 / fp32(d))), -31, 31) (0 when d is 0), y = q x fp32(d): what the journal would return for
// these values (the append's block quantizer and the seal's dequantizer, operation for
// operation).
__device__ __forceinline__ void tq6_roundtrip(float (&y)[128]) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 128; ++i) a = fmaxf(a, fabsf(y[i]));
    const float d = h2f(f2h_bits(fdiv(a, 31.0f)));
    const float inv = (d == 0.f) ? 0.f : fdiv(1.0f, d);
    const float2 inv2 = make_float2(inv, inv), d2 = make_float2(d, d);
#pragma unroll
    for (int i = 0; i < 128; i += 2) {
        const float2 t = fmul2(make_float2(y[i], y[i + 1]), inv2);
        float2 q = make_float2((d == 0.f) ? 0.f : rintf(t.x), (d == 0.f) ? 0.f : rintf(t.y));
        q = make_float2(fminf(fmaxf(q.x, -31.f), 31.f), fminf(fmaxf(q.y, -31.f), 31.f));
        const float2 r = fmul2(q, d2);
        y[i] = r.x; y[i + 1] = r.y;
    }
}

// Row t of a staged tq6_0 tile: y_i = (code_i - 32) x fp32(d), an exact product.
// A 32-bit word of the ql plane holds 8 channels' low nibbles; the matching 16 bits of the
// qh plane their 2-bit high parts, spread here so that each channel's pair lands in bits
// 4-5 of the byte that holds its nibble. A byte c placed in bits 8-15 under exponent 15
// reads as the float f = 2^15 + c, and y = fma(f, d, -(2^15 + 32) d): the addend is exact
// ((2^15 + 32) = 32 x 1025 has 11 significant bits, d at most 11) and so is the result, the
// representable (c - 32) d, whatever the rounding. (A non-finite d, which only non-finite
// inputs produce and the status word flags, gives NaN rows here.)
__device__ __forceinline__ void decode_tq6(const uint8_t* st, int D, int b, float (&y)[128]) {
    const int t = threadIdx.x;
    const uint4* rp = reinterpret_cast<const uint4*>(st + t * kTq6Stride);
    uint32_t q[16], h[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 x = rp[i];
        q[4 * i] = x.x; q[4 * i + 1] = x.y; q[4 * i + 2] = x.z; q[4 * i + 3] = x.w;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint4 x = rp[4 + i];
        h[4 * i] = x.x; h[4 * i + 1] = x.y; h[4 * i + 2] = x.z; h[4 * i + 3] = x.w;
    }
    const float d = h2f(reinterpret_cast<const uint16_t*>(st + kRows * kTq6Stride)[t * (D / 128) + b]);
    const float a = fmul(-32800.0f, d);
    const float2 d2 = make_float2(d, d), a2 = make_float2(a, a);
#pragma unroll
    for (int w = 0; w < 16; ++w) {
        uint32_t x = (w & 1) ? (h[w >> 1] >> 16) : (h[w >> 1] & 0xFFFFu);
        x = (x | (x << 8)) & 0x00FF00FFu;
        x = (x | (x << 4)) & 0x0F0F0F0Fu;
        x = (x | (x << 2)) & 0x33333333u;     // channel 8w + e: high pair at bits 4e, 4e + 1
        const uint32_t ev = (q[w] & 0x0F0F0F0Fu) | ((x << 4) & 0xF0F0F0F0u);   // channels 8w + 2k
        const uint32_t od = ((q[w] >> 4) & 0x0F0F0F0Fu) | (x & 0xF0F0F0F0u);   // channels 8w + 2k + 1
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float ce = __uint_as_float(__byte_perm(ev, 0x47000000u, 0x7404 + 16 * k));
            const float co = __uint_as_float(__byte_perm(od, 0x47000000u, 0x7404 + 16 * k));
            const float2 v = ffma2(make_float2(ce, co), d2, a2);
            y[8 * w + 2 * k] = v.x;
            y[8 * w + 2 * k + 1] = v.y;
        }
    }
}

// Row t of a staged 16-bit tile, widened exactly.
template <int JK>
__device__ __forceinline__ void decode_x16(const uint8_t* st, float (&y)[128]) {
    const uint4* rp = reinterpret_cast<const uint4*>(st + threadIdx.x * kX16Stride);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint4 x = rp[i];
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = 8 * i + 2 * k;
            if constexpr (JK == J_BF16) {
                y[j] = __uint_as_float(wv[k] << 16);
                y[j + 1] = __uint_as_float(wv[k] & 0xFFFF0000u);
            } else {
                y[j] = h2f((uint16_t)(wv[k] & 0xFFFFu));
                y[j + 1] = h2f((uint16_t)(wv[k] >> 16));
            }
        }
    }
}

// TBQ128 of one 128-channel block in registers: s2 . FWHT_128(s1 . x) x fp32(1/sqrt(128)),
// butterflies in ascending stride order (the same operations as any other FWHT of the codec).
// Strides 2 .. 64 go two butterflies (i, i + 1) per instruction pair; their inputs are sums
// or the staged values, never products.
__device__ __forceinline__ void rotate_tbq128(float (&y)[128]) {
#pragma unroll
    for (int i = 0; i < 128; ++i)
        if (sign_neg(0, i)) y[i] = -y[i];
#pragma unroll
    for (int i = 0; i < 128; i += 2) {
        const float a = y[i], c = y[i + 1];
        y[i] = fadd(a, c);
        y[i + 1] = fsub(a, c);
    }
#pragma unroll
    for (int s = 2; s < 128; s <<= 1) {
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
            if (i & s) continue;
            const float2 a = make_float2(y[i], y[i + 1]), c = make_float2(y[i + s], y[i + s + 1]);
            const float2 u = fadd2(a, c), v = fsub2(a, c);
            y[i] = u.x; y[i + 1] = u.y;
            y[i + s] = v.x; y[i + s + 1] = v.y;
        }
    }
#pragma unroll
    for (int i = 0; i < 128; i += 2) {
        const float2 v = make_float2(sign_neg(1, i) ? -y[i] : y[i], sign_neg(1, i + 1) ? -y[i + 1] : y[i + 1]);
        const float2 r = fmul2(v, make_float2(kTbqScale, kTbqScale));
        y[i] = r.x; y[i + 1] = r.y;
    }
}

// ---------------------------------------------------------------------------- encoders
// The halving tree of y_i^2 over 128 values: node(0, i) = y_i^2 and node(K, i) = node(K-1, i)
// + node(K-1, i + 128 / 2^K); node(7, 0) is the sum. Nodes (K, I) and (K, I + 1) go as one
// pair (I even, K <= 6: the partner offset 128 / 2^K is even, so the two nodes' terms pair up
// level by level), evaluated depth first so that few partial sums are live beside the 128
// values. The leaves are fma(y_i, y_i, z) with z a run-time +0 the code generator cannot fold:
// exactly y_i^2 (a square is never -0), and a multiply-add result, which no later add can be
// contracted with (a packed multiply feeding the packed adds could be).
template <int K, int I>
__device__ __forceinline__ float2 sq_tree2(const float (&y)[128], float2 z) {
    if constexpr (K == 0) {
        const float2 v = make_float2(y[I], y[I + 1]);
        return ffma2(v, v, z);
    } else {
        return fadd2(sq_tree2<K - 1, I>(y, z), sq_tree2<K - 1, I + (128 >> K)>(y, z));
    }
}
// node (7, 0) = node (6, 0) + node (6, 1)
__device__ __forceinline__ float sq_sum128(const float (&y)[128], float zero) {
    const float2 p = sq_tree2<6, 0>(y, make_float2(zero, zero));
    return fadd(p.x, p.y);
}

// Order-preserving integer key of an fp32 value: its bits for +0 and above, its bits with the 31
// magnitude bits inverted for negative values. Within one sign the key grows with the value.
__device__ __forceinline__ uint32_t fkey(float x) {
    const uint32_t b = __float_as_uint(x);
    return b ^ ((uint32_t)((int32_t)b >> 31) >> 1);
}

// The bits b of a value as a 32-bit integer's absolute value: b for +0 and above, 2^32 - b for
// negative values (2^31 for -0: abs.s32 keeps the most negative integer). For those it is
// fkey(b) + 2^31 + 1 (mod 2^32), which the negative buckets' table entries absorb.
__device__ __forceinline__ uint32_t iabs_bits(uint32_t b) {
    uint32_t r;
    asm("abs.s32 %0, %1;" : "=r"(r) : "r"(b));
    return r;
}

// TBQ4 block: n16 = fp16(sqrt(sum y^2)), u = y x (1 / fp32(n16)) (0 when n16 is 0), idx =
// #{k : u > beta_k}; nibble e of P[m] is the index of channel 8m + e. The table entry of the
// bucket of u's bits plus iabs_bits(u) has the index in its top four bits (build_qtab); a
// funnel shift moves it into the packed word (channel 8m + 7 first, so that channel 8m ends
// in nibble 0).
__device__ __forceinline__ uint16_t encode_tbq4(const float (&y)[128], const uint32_t* qt, uint32_t (&P)[16],
                                               float zero) {
    const uint16_t n16 = f2h_bits(__fsqrt_rn(sq_sum128(y, zero)));
    const float n = h2f(n16);
    const float inv = (n == 0.f) ? 0.f : fdiv(1.0f, n);
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        uint32_t acc = 0;
#pragma unroll
        for (int e = 6; e >= 0; e -= 2) {
            const float2 u = fmul2(make_float2(y[8 * m + e], y[8 * m + e + 1]), inv2);
            const uint32_t b1 = __float_as_uint(u.y), b0 = __float_as_uint(u.x);
            acc = __funnelshift_l(qt[b1 >> 21] + iabs_bits(b1), acc, 4);
            acc = __funnelshift_l(qt[b0 >> 21] + iabs_bits(b0), acc, 4);
        }
        P[m] = acc;
    }
    return n16;
}

// Q8_0 (QMAX 127) or Q4_0 (QMAX 7) block of 32 values starting at channel j0: d = fp16(max|x|
// / QMAX), q = clamp(rint(x x (1 / fp32(d))), -QMAX, QMAX) (inv 0 when d is 0). The clamp is
// taken before the rounding, which gives the same integer for an integer QMAX; adding
// 1.5 x 2^23 (+ 8, the Q4_0 zero point) rounds half to even and leaves the code in the low
// byte. c[k] holds the code bytes of channels j0 + 4k .. j0 + 4k + 3.
template <int QMAX>
__device__ __forceinline__ uint16_t encode_q32(const float (&y)[128], int j0, uint32_t (&c)[8]) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(y[j0 + i]));
    const uint16_t d16 = f2h_bits(fdiv(a, (float)QMAX));
    const float d = h2f(d16);
    const float inv = (d == 0.f) ? 0.f : fdiv(1.0f, d);
    // 1.5 x 2^23 plus the zero level (Q8_0: 0, its codes are signed bytes; else QMAX + 1)
    constexpr float magic = 12582912.0f + (QMAX == 127 ? 0.f : (float)(QMAX + 1));
    const float2 inv2 = make_float2(inv, inv), mg2 = make_float2(magic, magic);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; i += 2) {   // the clamp stands between the packed multiply and add
            const float2 t = fmul2(make_float2(y[j0 + 4 * k + i], y[j0 + 4 * k + i + 1]), inv2);
            const float2 z = make_float2(fminf(fmaxf(t.x, -(float)QMAX), (float)QMAX),
                                         fminf(fmaxf(t.y, -(float)QMAX), (float)QMAX));
            const float2 v = fadd2(z, mg2);
            r[i] = __float_as_uint(v.x);
            r[i + 1] = __float_as_uint(v.y);
        }
        c[k] = __byte_perm(__byte_perm(r[0], r[1], 0x0040), __byte_perm(r[2], r[3], 0x0040), 0x5410);
    }
    return d16;
}

// Q4_1 (Q 15) or Q5_1 (Q 31) block of 32 values starting at channel j0: m = fp16(min x),
// d = fp16((max x - min x) / Q), code = clamp(rint((x - fp32(m)) x (1 / fp32(d))), 0, Q) (inv 0
// when d is 0), rounded by adding 1.5 x 2^23. c[k] holds the code bytes of channels j0 + 4k ..
template <int Q>
__device__ __forceinline__ uint16_t encode_qmin(const float (&y)[128], int j0, uint32_t (&c)[8], uint16_t& m16) {
    float lo = y[j0], hi = y[j0];
#pragma unroll
    for (int i = 1; i < 32; ++i) {
        lo = fminf(lo, y[j0 + i]);
        hi = fmaxf(hi, y[j0 + i]);
    }
    m16 = f2h_bits(lo);
    const uint16_t d16 = f2h_bits(fdiv(fsub(hi, lo), (float)Q));
    const float d = h2f(d16), m = h2f(m16);
    const float inv = (d == 0.f) ? 0.f : fdiv(1.0f, d);
    const float2 m2 = make_float2(m, m), inv2 = make_float2(inv, inv), mg2 = make_float2(12582912.0f, 12582912.0f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; i += 2) {   // the clamp stands between the packed multiply and add
            const float2 t = fmul2(fsub2(make_float2(y[j0 + 4 * k + i], y[j0 + 4 * k + i + 1]), m2), inv2);
            const float2 v = fadd2(make_float2(fminf(fmaxf(t.x, 0.f), (float)Q), fminf(fmaxf(t.y, 0.f), (float)Q)), mg2);
            r[i] = __float_as_uint(v.x);
            r[i + 1] = __float_as_uint(v.y);
        }
        c[k] = __byte_perm(__byte_perm(r[0], r[1], 0x0040), __byte_perm(r[2], r[3], 0x0040), 0x5410);
    }
    return d16;
}

// Bit 4 of 8 code bytes (two words, channels 8m .. 8m + 7) as one byte, channel e at bit e:
// the multiply gathers the bits at 0, 8, 16, 24 into bits 21 .. 24 (no two partial products meet).
__device__ __forceinline__ uint32_t bit4_byte(uint32_t c0, uint32_t c1) {
    const uint32_t a = (c0 >> 4) & 0x01010101u, b = (c1 >> 4) & 0x01010101u;
    return (((a * 0x00204081u) >> 21) & 0xFu) | ((((b * 0x00204081u) >> 21) & 0xFu) << 4);
}
// Bits 4-5 of 4 code bytes (one word, channels 4m .. 4m + 3) as one byte, channel e at bits 2e.
__device__ __forceinline__ uint32_t bits45_byte(uint32_t c) {
    const uint32_t a = (c >> 4) & 0x03030303u;
    return ((a * 0x00041041u) >> 18) & 0xFFu;
}

// Two words of code bytes (8 channels, values < 16) as one word of nibbles, the even channel
// in the low nibble.
__device__ __forceinline__ uint32_t nibbles_of(uint32_t c0, uint32_t c1) {
    return __byte_perm(c0 | (c0 >> 4), c1 | (c1 >> 4), 0x6420);
}

// 8 x 8 transpose of nibbles inside groups of 8 lanes: lane j holds row j (nibble e =
// column e) on entry and column j (nibble i = row i) on exit. Block swaps of 4 x 4 (16-bit
// halves), 2 x 2 (bytes) and 1 x 1 (nibbles).
__device__ __forceinline__ uint32_t transpose_nib8(uint32_t x, int lane) {
    uint32_t y = __shfl_xor_sync(kFull, x, 4);
    x = __byte_perm(x, y, (lane & 4) ? 0x3276 : 0x5410);
    y = __shfl_xor_sync(kFull, x, 2);
    x = __byte_perm(x, y, (lane & 2) ? 0x3715 : 0x6240);
    y = __shfl_xor_sync(kFull, x, 1);
    y = __funnelshift_l(y, y, (lane & 1) ? 28 : 4);
    const uint32_t keep = (lane & 1) ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
    return (x & keep) | (y & ~keep);
}

// 4 x 4 transpose of bytes inside groups of 4 lanes (the same block swaps).
__device__ __forceinline__ uint32_t transpose_byte4(uint32_t x, int lane) {
    uint32_t y = __shfl_xor_sync(kFull, x, 2);
    x = __byte_perm(x, y, (lane & 2) ? 0x3276 : 0x5410);
    y = __shfl_xor_sync(kFull, x, 1);
    return __byte_perm(x, y, (lane & 1) ? 0x3715 : 0x6240);
}

// 4-bit codes of row t, block b: K rows of D/2 bytes; V channel rows of 64 bytes.
__device__ __forceinline__ void store_nibbles(uint8_t* rec, int D, int b, int w, const uint32_t (&P)[16]) {
    const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
    if (w == 0) {
        uint4* dst = reinterpret_cast<uint4*>(rec + (int64_t)t * (D / 2) + 64 * b);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(P[4 * i], P[4 * i + 1], P[4 * i + 2], P[4 * i + 3]);
    } else {
        // lane 8a + e ends with channel 8m + e of positions 32 wp + 8a .. + 7
        uint8_t* base = rec + (int64_t)(128 * b + (lane & 7)) * 64 + 16 * wp + 4 * (lane >> 3);
#pragma unroll
        for (int m = 0; m < 16; ++m)
            *reinterpret_cast<uint32_t*>(base + 8 * m * 64) = transpose_nib8(P[m], lane);
    }
}

// Q8_0 codes of row t, block b: K rows of D bytes; V channel rows of 128 bytes.
__device__ __forceinline__ void store_bytes(uint8_t* rec, int D, int b, int w, const uint32_t (&B)[32]) {
    const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
    if (w == 0) {
        uint4* dst = reinterpret_cast<uint4*>(rec + (int64_t)t * D + 128 * b);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_uint4(B[4 * i], B[4 * i + 1], B[4 * i + 2], B[4 * i + 3]);
    } else {
        // lane 4a + e ends with channel 4m + e of positions 32 wp + 4a .. + 3
        uint8_t* base = rec + (int64_t)(128 * b + (lane & 3)) * 128 + 32 * wp + 4 * (lane >> 2);
#pragma unroll
        for (int m = 0; m < 32; ++m)
            *reinterpret_cast<uint32_t*>(base + 4 * m * 128) = transpose_byte4(B[m], lane);
    }
}

// Decision table of a TBQ index (TBQ4: the 15 boundaries; turbo3: 7) over keys (fkey): bucket k
// = the values whose key has top 11 bits k, a value range [vmin, vmax]. base = boundaries below
// vmin; thr = the boundary inside the bucket, if any, as the low 21 bits t of the largest key
// in the bucket whose value does not exceed it (the key of the boundary itself; for the zero
// boundary in the bucket of -0, the bucket's largest key, which no value of the bucket exceeds);
// without one t = 0x1FFFFF. Entry = (base << 28) + (2^28 - 1 - t) - (k << 21), so that for a key
// x of the bucket the sum entry + x = (base << 28) + 2^28 - 1 - t + (x & 0x1FFFFF) carries into
// bit 28 exactly when x & 0x1FFFFF > t, i.e. when u > thr: (entry + x) >> 28 = base + (u > thr)
// (never above 15: a bucket with a boundary has base <= 14). Buckets of infinities and NaNs
// give 0 (a NaN exceeds no boundary). Exact where no bucket holds two boundaries (consecutive
// boundaries differ by a ratio above 1.25: TBQ4 >= 1.28, turbo3 >= 1.66).
// The kernel indexes the table by u's own top 11 bits and adds iabs_bits(u) (encode_tbq4): the
// entry of key bucket k of a negative value is stored at index k ^ 0x3FF (its bits' bucket)
// and raised by 2^31 - 1, fkey(u) minus iabs_bits(u) (mod 2^32).
__device__ void build_qtab(uint32_t* qt, const float* bnd, int nb) {
    for (int k = threadIdx.x; k < kBuckets; k += blockDim.x) {
        const uint32_t klo = (uint32_t)k << 21, khi = klo | 0x1FFFFFu;
        const bool neg = k >= kBuckets / 2;
        const uint32_t flip = neg ? 0x7FFFFFFFu : 0u;
        const uint32_t blo = klo ^ flip, bhi = khi ^ flip;   // bits of the smallest and largest value
        uint32_t t = 0x1FFFFFu, base = 0;
        if (((blo >> 23) & 0xFF) != 0xFF) {
            const float vmin = __uint_as_float(blo), vmax = __uint_as_float(bhi);
            for (int j = 0; j < nb; ++j) {
                const float bj = bnd[j];
                if (bj < vmin) ++base;
                else if (bj <= vmax) t = (neg && bj == 0.f) ? 0x1FFFFFu : (fkey(bj) & 0x1FFFFFu);
            }
        }
        qt[neg ? (k ^ 0x3FF) : k] = (base << 28) + (0x0FFFFFFFu - t) - klo + (neg ? 0x7FFFFFFFu : 0u);
    }
}

// tq5_0 block (128 values): d = fp16(max|y| / 15), code = clamp(rint(y x (1 / fp32(d))), -15, 15)
// + 16 (inv 0 when d is 0), rounded by adding 1.5 x 2^23 + 16; c[k] holds the code bytes of
// channels 4k .. 4k + 3.
__device__ __forceinline__ uint16_t encode_tq5(const float (&y)[128], uint32_t (&c)[32]) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 128; ++i) a = fmaxf(a, fabsf(y[i]));
    const uint16_t d16 = f2h_bits(fdiv(a, 15.0f));
    const float d = h2f(d16);
    const float inv = (d == 0.f) ? 0.f : fdiv(1.0f, d);
    const float2 inv2 = make_float2(inv, inv), mg2 = make_float2(12582928.0f, 12582928.0f);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        uint32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; i += 2) {   // the clamp stands between the packed multiply and add
            const float2 t = fmul2(make_float2(y[4 * k + i], y[4 * k + i + 1]), inv2);
            const float2 v = fadd2(make_float2(fminf(fmaxf(t.x, -15.f), 15.f), fminf(fmaxf(t.y, -15.f), 15.f)), mg2);
            r[i] = __float_as_uint(v.x);
            r[i + 1] = __float_as_uint(v.y);
        }
        c[k] = __byte_perm(__byte_perm(r[0], r[1], 0x0040), __byte_perm(r[2], r[3], 0x0040), 0x5410);
    }
    return d16;
}

// The low two bits of 8 nibbles (channels 8m .. 8m + 7) as 16 bits, channel e at bits 2e.
__device__ __forceinline__ uint32_t crumbs_of(uint32_t x) {
    x &= 0x33333333u;
    x = (x | (x >> 2)) & 0x0F0F0F0Fu;
    x = (x | (x >> 4)) & 0x00FF00FFu;
    return (x | (x >> 8)) & 0x0000FFFFu;
}
// Bit 2 of 8 nibbles as one byte, channel e at bit e.
__device__ __forceinline__ uint32_t bit2_byte(uint32_t x) {
    x = (x >> 2) & 0x11111111u;
    x = (x | (x >> 3)) & 0x03030303u;
    x = (x | (x >> 6)) & 0x000F000Fu;
    return (x | (x >> 12)) & 0xFFu;
}

// ---------------------------------------------------------------------------- kernel
// One instance per journal kind and body family: TBQ4 layouts (K and V TBQ4: the rotation
// is per layout) or Q8_0 / Q4_0 layouts, so that each instance holds one encoder's code.
// The pure instances (F_TBQ4_ONLY: TBQ4 keys and values; F_Q84: Q8_0 / Q4_0 keys and values)
// compile only their own encoders, which keeps the kernel's code, and its instruction-cache
// misses, small for the layouts the workloads use.
enum BodyFamily { F_TBQ4 = 0, F_Q = 1, F_TBQ4_ONLY = 2, F_Q84 = 3 };
template <int FAM> constexpr bool kRotFam = FAM == F_TBQ4 || FAM == F_TBQ4_ONLY;

// Decodes the tiles of iterations k0 .. k0 + kSlotBatch - 1 into the slot ring (threads 4j).
__device__ __forceinline__ void fill_slots(const Layout& L, const SealParams& p, int n_tiles, TileSlot* slot, int k0) {
    const int t = threadIdx.x;
    if ((t & 3) == 0) {
        const int k = k0 + (t >> 2);
        const int tile = blockIdx.x + k * gridDim.x;
        if (tile < n_tiles) slot[k % kSlots] = tile_slot(L, p, tile);
    }
}

template <int JK, int FAM>
__global__ void __launch_bounds__(kRows, JK == J_TQ6 ? 3 : 2)
seal_rows_kernel(Layout L, SealParams p, int n_tiles, int stage_bytes, float zero) {
    extern __shared__ __align__(16) uint8_t sm[];
    __shared__ TileSlot slot[kSlots];
    uint32_t* qt = reinterpret_cast<uint32_t*>(sm + kStages * stage_bytes);
    uint32_t* qt3 = qt + kBuckets;                  // turbo3's table, present when a body is turbo3
    if constexpr (kRotFam<FAM>) {                   // read after the first barrier below
        build_qtab(qt, c_tab.bnd, 15);
        if (FAM == F_TBQ4 && (L.fmt[0] == KVQ_TURBO3 || L.fmt[1] == KVQ_TURBO3)) build_qtab(qt3, c_tab.bnd3, 7);
    }
    const int t = threadIdx.x, D = L.D;
    // Iteration it encodes tile blockIdx.x + it * gridDim.x from stage it % kStages. After the
    // iteration's barrier every thread has finished iteration it - 1, so its stage takes tile
    // it + kStages - 1 and the slots it read may be rewritten.
    fill_slots(L, p, n_tiles, slot, 0);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
        if ((int)blockIdx.x + k * (int)gridDim.x < n_tiles) issue_tile<JK>(L, slot[k], sm + k * stage_bytes);
        cp_async_commit();
    }
    for (int it = 0;; ++it) {
        const int tile = blockIdx.x + it * gridDim.x;
        if (tile >= n_tiles) break;
        cp_async_wait<kStages - 2>();   // this thread's copies of tile `it` have landed
        __syncthreads();                // and everyone else's; iteration it - 1 is done
        const int ahead = it + kStages - 1;
        if (tile + (kStages - 1) * (int)gridDim.x < n_tiles)
            issue_tile<JK>(L, slot[ahead % kSlots], sm + (ahead % kStages) * stage_bytes);
        cp_async_commit();
        // slots of iterations it + kStages .. (read from iteration it + 1 on) while the ring
        // holds it .. it + kStages - 1
        if (it % kSlotBatch == 0) fill_slots(L, p, n_tiles, slot, it + kStages);

        const TileSlot tl = slot[it % kSlots];
        const uint8_t* st = sm + (it % kStages) * stage_bytes;
        float y[128];
        if constexpr (JK == J_TQ6) {
            decode_tq6(st, D, tl.b, y);
        } else if constexpr (JK == J_IN) {
            // a prefill chunk's fp16 rows, turned into what the journal would hold for them: the
            // stored 16-bit values (bf16-rounded for a BF16 journal), rotated; with a tq6_0 ring
            // the rotated rows are staged and dequantized
            decode_x16<J_F16>(st, y);
            if (L.journal == KVQ_BF16) {
#pragma unroll
                for (int i = 0; i < 128; ++i) y[i] = bf2f(f2bf_bits(y[i]));
            }
            if constexpr (kRotFam<FAM>) rotate_tbq128(y);
            if (L.journal == KVQ_TQ6_0) tq6_roundtrip(y);
        } else {
            decode_x16<JK>(st, y);
            if constexpr (kRotFam<FAM>) rotate_tbq128(y);
        }
        uint8_t* rec = tl.rec;
        const int fmt = L.fmt[tl.w];
        if constexpr (kRotFam<FAM>) {
            if (FAM == F_TBQ4 && fmt == KVQ_TQ5_0) {   // token-major: nibble plane, one-bit plane, scales
                uint32_t C[32], P[16], hb[4];
                const uint16_t d16 = encode_tq5(y, C);
#pragma unroll
                for (int m = 0; m < 16; ++m) P[m] = nibbles_of(C[2 * m] & 0x0F0F0F0Fu, C[2 * m + 1] & 0x0F0F0F0Fu);
                store_nibbles(rec, D, tl.b, 0, P);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    hb[q] = bit4_byte(C[8 * q], C[8 * q + 1]) | (bit4_byte(C[8 * q + 2], C[8 * q + 3]) << 8) |
                            (bit4_byte(C[8 * q + 4], C[8 * q + 5]) << 16) | (bit4_byte(C[8 * q + 6], C[8 * q + 7]) << 24);
                *reinterpret_cast<uint4*>(rec + 64LL * D + (int64_t)t * (D / 8) + 16 * tl.b) =
                    make_uint4(hb[0], hb[1], hb[2], hb[3]);
                reinterpret_cast<uint16_t*>(rec + 80LL * D)[t * (D / 128) + tl.b] = d16;
                flag_nonfinite(L, p.pool, h2f(d16));
            } else {
                uint32_t P[16];
                const bool t3 = FAM == F_TBQ4 && fmt == KVQ_TURBO3;
                const uint16_t n16 = encode_tbq4(y, t3 ? qt3 : qt, P, zero);
                if (t3) {   // token-major: 2-bit plane, one-bit plane, norms
                    uint32_t cw[8], bw[4];
#pragma unroll
                    for (int q = 0; q < 8; ++q) cw[q] = crumbs_of(P[2 * q]) | (crumbs_of(P[2 * q + 1]) << 16);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        bw[q] = bit2_byte(P[4 * q]) | (bit2_byte(P[4 * q + 1]) << 8) | (bit2_byte(P[4 * q + 2]) << 16) |
                                (bit2_byte(P[4 * q + 3]) << 24);
                    uint4* c2 = reinterpret_cast<uint4*>(rec + (int64_t)t * (D / 4) + 32 * tl.b);
                    c2[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    c2[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                    *reinterpret_cast<uint4*>(rec + 32LL * D + (int64_t)t * (D / 8) + 16 * tl.b) =
                        make_uint4(bw[0], bw[1], bw[2], bw[3]);
                    reinterpret_cast<uint16_t*>(rec + 48LL * D)[t * (D / 128) + tl.b] = n16;
                } else {
                    store_nibbles(rec, D, tl.b, tl.w, P);
                    reinterpret_cast<uint16_t*>(rec + 64LL * D)[t * (D / 128) + tl.b] = n16;
                }
                flag_nonfinite(L, p.pool, h2f(n16));
            }
        } else {
            uint16_t d16[4], m16[4] = {0, 0, 0, 0};
            uint32_t C[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t c[8];
                if constexpr (FAM == F_Q84) {
                    if (fmt == KVQ_Q8_0) d16[j] = encode_q32<127>(y, 32 * j, c);
                    else d16[j] = encode_q32<7>(y, 32 * j, c);
                } else {
                    switch (fmt) {
                        case KVQ_Q8_0: d16[j] = encode_q32<127>(y, 32 * j, c); break;
                        case KVQ_Q4_0: d16[j] = encode_q32<7>(y, 32 * j, c); break;
                        case KVQ_Q5_0: d16[j] = encode_q32<15>(y, 32 * j, c); break;
                        case KVQ_Q6_0: d16[j] = encode_q32<31>(y, 32 * j, c); break;
                        case KVQ_Q4_1: d16[j] = encode_qmin<15>(y, 32 * j, c, m16[j]); break;
                        default: d16[j] = encode_qmin<31>(y, 32 * j, c, m16[j]); break;
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) C[8 * j + k] = c[k];
            }
            const int qbits = (FAM == F_Q84) ? 0 : qblock_bits(fmt);
            int64_t sc_off;
            if (fmt == KVQ_Q8_0) {
                store_bytes(rec, D, tl.b, tl.w, C);
                sc_off = 128LL * D;
            } else {
                // Q4_0: K token-major, V channel-major; the other block formats token-major for
                // both, the low nibbles then the high plane of the 5- and 6-bit codes
                uint32_t P[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) P[m] = nibbles_of(C[2 * m] & 0x0F0F0F0Fu, C[2 * m + 1] & 0x0F0F0F0Fu);
                store_nibbles(rec, D, tl.b, qbits ? 0 : tl.w, P);
                if (qbits == 5) {
                    uint32_t hb[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        hb[q] = bit4_byte(C[8 * q], C[8 * q + 1]) | (bit4_byte(C[8 * q + 2], C[8 * q + 3]) << 8) |
                                (bit4_byte(C[8 * q + 4], C[8 * q + 5]) << 16) | (bit4_byte(C[8 * q + 6], C[8 * q + 7]) << 24);
                    *reinterpret_cast<uint4*>(rec + 64LL * D + (int64_t)t * (D / 8) + 16 * tl.b) =
                        make_uint4(hb[0], hb[1], hb[2], hb[3]);
                } else if (qbits == 6) {
                    uint32_t hb[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        hb[q] = bits45_byte(C[4 * q]) | (bits45_byte(C[4 * q + 1]) << 8) | (bits45_byte(C[4 * q + 2]) << 16) |
                                (bits45_byte(C[4 * q + 3]) << 24);
                    uint4* dst = reinterpret_cast<uint4*>(rec + 64LL * D + (int64_t)t * (D / 4) + 32 * tl.b);
                    dst[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
                    dst[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
                }
                sc_off = record_code_bytes(fmt, D);
            }
            *reinterpret_cast<uint2*>(rec + sc_off + 2LL * (t * (D / 32) + 4 * tl.b)) =
                make_uint2(d16[0] | ((uint32_t)d16[1] << 16), d16[2] | ((uint32_t)d16[3] << 16));
            if (qbits && qblock_sym_levels(fmt) == 0) {
                *reinterpret_cast<uint2*>(rec + sc_off + 8LL * D + 2LL * (t * (D / 32) + 4 * tl.b)) =
                    make_uint2(m16[0] | ((uint32_t)m16[1] << 16), m16[2] | ((uint32_t)m16[3] << 16));
#pragma unroll
                for (int j = 0; j < 4; ++j) flag_nonfinite(L, p.pool, h2f(m16[j]));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) flag_nonfinite(L, p.pool, h2f(d16[j]));
        }
    }
}

template <int JK, int FAM>
int launch_rows(const Layout& L, const SealParams& p, int n_tiles, cudaStream_t s) {
    const int stage = (JK == J_TQ6) ? kRows * kTq6Stride + 2 * L.D : kRows * kX16Stride;
    const bool t3 = (L.fmt[0] == KVQ_TURBO3 || L.fmt[1] == KVQ_TURBO3);
    const size_t smem = (size_t)kStages * stage + (kRotFam<FAM> ? (t3 ? 2 : 1) * kBuckets * sizeof(uint32_t) : 0);
    auto fn = seal_rows_kernel<JK, FAM>;
    int e = (int)cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e) return e;
    int per_sm = 0, dev = 0;
    e = (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kRows, smem);
    if (e) return e;
    e = (int)cudaGetDevice(&dev);
    if (e) return e;
    const int grid = std::min(n_tiles, std::max(per_sm, 1) * query_sm_count(dev));
    fn<<<grid, kRows, smem, s>>>(L, p, n_tiles, stage, 0.0f);   // zero: see sq_tree2
    return (int)cudaGetLastError();
}

template <int FAM>
int launch_family(const Layout& L, const SealParams& p, int n_tiles, cudaStream_t s) {
    if (p.k_src != nullptr) return launch_rows<J_IN, FAM>(L, p, n_tiles, s);
    if (L.journal == KVQ_TQ6_0) return launch_rows<J_TQ6, FAM>(L, p, n_tiles, s);
    if (L.journal == KVQ_BF16) return launch_rows<J_BF16, FAM>(L, p, n_tiles, s);
    return launch_rows<J_F16, FAM>(L, p, n_tiles, s);
}

// ---------------------------------------------------------------------------- KVarN seal
// One 128 x 256 tile (SJ-KVaRN §2.2): HAD256-rotated journal rows, 16 alternating row/column
// passes of spread balancing (rows first), per-row b-bit rounding with fp16 scales (SJ-KVaRN
// §2.2, §3). CTA = 16 warps on one tile = (group, KV head, K or V, 256-channel half). The
// tile's journal rows are staged once with cp.async and decoded from shared memory twice (into
// the balanced tile, and again for the codes, which use the unbalanced values). The balanced
// tile lives in registers: thread (warp w, lane l) holds the 64 values of rows w + 16 a and
// columns l + 32 b (a, b < 8). A line's halving-tree sums take their first three levels in the
// thread (value pairs a, a + 4 / a, a + 2 / a, a + 1, likewise for b); the last five levels of
// a row cross the warp's lanes (shuffles), the last four of a column cross the 16 warps through
// 16 KB of shared memory. So a pass moves partial sums, not the tile. The arithmetic is the
// codec's, operation for operation.
constexpr int kKvThreads = 512;
constexpr int kKvWarps = kKvThreads / 32;

template <int JK>
struct KvStage {
    static constexpr int ROW = (JK == J_TQ6) ? 192 : 512;    // one row of the half (2 tq6_0 blocks / 256 x 16 bit)
};

// The tq6_0 staging of one 128-value block held by a warp, 4 values per lane (v[k0 .. k0+3]), in
// place: the same arithmetic as tq6_roundtrip.
__device__ __forceinline__ void tq6_roundtrip_warp(float (&v)[8], int k0) {
    float a = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) a = fmaxf(a, fabsf(v[k0 + m]));
    a = warp_max(a);
    const float d = h2f(f2h_bits(fdiv(a, 31.0f)));
    const float inv = (d == 0.f) ? 0.f : fdiv(1.0f, d);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        float q = (d == 0.f) ? 0.f : rintf(fmul(v[k0 + m], inv));
        q = fminf(fmaxf(q, -31.f), 31.f);
        v[k0 + m] = fmul(q, d);
    }
}

// Values of channels lane + 32k (k < 8) of row t of the staged half, in the body's domain:
// tq6_0 codes dequantized (the ring rows are rotated at append), 16-bit rows widened and
// rotated here by HAD256.
template <int JK>
__device__ __forceinline__ void kv_row(const uint8_t* st, const uint16_t* sc, int t, int nsc, int half, int lane,
                                       float (&v)[8], int journal, float nz) {
    const uint8_t* row = st + t * KvStage<JK>::ROW;
    if constexpr (JK == J_IN) {
        // a prefill chunk's fp16 row: the stored value (bf16-rounded for a BF16 journal),
        // rotated, and with a tq6_0 ring staged and dequantized per 128-channel block
        const uint16_t* r16 = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            v[k] = h2f(r16[lane + 32 * k]);
            if (journal == KVQ_BF16) v[k] = bf2f(f2bf_bits(v[k]));
        }
        warp_fwht<8>(v, lane);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __fmaf_rn(v[k], kHad256Scale, nz);
        if (journal == KVQ_TQ6_0) {
            tq6_roundtrip_warp(v, 0);
            tq6_roundtrip_warp(v, 4);
        }
    } else if constexpr (JK == J_TQ6) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int b = k >> 2, j = lane + 32 * (k & 3);
            const uint8_t* blk = row + 96 * b;
            const int lo = (blk[j >> 1] >> ((j & 1) * 4)) & 15;
            const int hi = (blk[64 + (j >> 2)] >> ((j & 3) * 2)) & 3;
            v[k] = __fmaf_rn((float)((lo | (hi << 4)) - 32), h2f(sc[t * nsc + 2 * half + b]), nz);
        }
    } else {
        const uint16_t* r16 = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = x16_to_f(r16[lane + 32 * k], JK == J_BF16 ? KVQ_BF16 : KVQ_F16);
        warp_fwht<8>(v, lane);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __fmaf_rn(v[k], kHad256Scale, nz);
    }
}

// The reduction of 8 per-row values (v[k]: row k of this thread's rows) over the warp's 32
// lanes in the order of a halving tree over lane positions (lane pairs l, l + 16, then l + 8,
// l + 4, l + 2, l + 1). In the first three levels each lane of a pair keeps the half of the
// rows its lane bit selects and adds the partner's partial of that half, so every lane ends
// with the total of row lane / 4 (row 4 (l & 16 ? 1 : 0) + 2 (l & 8 ? 1 : 0) + (l & 4 ? 1 : 0))
// after 9 shuffles. OP is commutative in its bits (fp32 add, min, max): both lanes of a pair
// compute the same value.
template <class OP>
__device__ __forceinline__ float warp_rows8(const float (&v)[8], int lane, OP op) {
    const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4;
    float y[4], z[2];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = op(h4 ? v[k + 4] : v[k], __shfl_xor_sync(kFull, h4 ? v[k] : v[k + 4], 16));
#pragma unroll
    for (int k = 0; k < 2; ++k) z[k] = op(h3 ? y[k + 2] : y[k], __shfl_xor_sync(kFull, h3 ? y[k] : y[k + 2], 8));
    float u = op(h2 ? z[1] : z[0], __shfl_xor_sync(kFull, h2 ? z[0] : z[1], 4));
    u = op(u, __shfl_xor_sync(kFull, u, 2));
    return op(u, __shfl_xor_sync(kFull, u, 1));
}
struct FAdd { __device__ float operator()(float a, float b) const { return fadd(a, b); } };
struct FMin { __device__ float operator()(float a, float b) const { return fminf(a, b); } };
struct FMax { __device__ float operator()(float a, float b) const { return fmaxf(a, b); } };

// The spread of a line from its two halving-tree sums, as a pass computes it: sigma =
// sqrt(var / n), sigma <= 2^-20 counts as 1.
__device__ __forceinline__ float kv_sigma(float var_sum, float inv_n) {
    const float sig = __fsqrt_rn(fmul(var_sum, inv_n));
    return sig <= 9.5367431640625e-07f ? 1.f : sig;     // 2^-20
}

// A row pass over the warp's 8 rows (n = 256: mean, population spread, row /= sigma, the row
// scale r[t] *= sigma). Row positions j = l + 32 b: the thread's levels pair b with b + 4
// (stride 128), b + 2 (64), b + 1 (32); warp_rows8 takes strides 16 .. 1. Returns |sigma - 1|
// of row w + 16 (lane / 4); with APPLY false the pass only measures. Columns 2k and 2k + 1 go
// as pairs, two operations per instruction. Every product that an add consumes is a packed
// multiply-add with nz, a run-time -0 the code generator cannot fold: a + b x -0 rounds like
// the product alone (signed zeros included), and a multiply-add result cannot be contracted
// with the add that follows (a packed multiply feeding a packed add could be).
template <bool APPLY = true>
__device__ __forceinline__ float kv_row_pass(float (&x)[8][8], float* r, int warp, int lane, float nz) {
    constexpr float INV_N = 1.0f / 256.0f;
    const float2 nz2 = make_float2(nz, nz);
    float p[8];
    // leaf(a, k): the leaves of columns 2k and 2k + 1 as a pair; (l0 + l4, l1 + l5) and
    // (l2 + l6, l3 + l7), then their pair sum and its two halves
    auto partials = [&](auto leaf) {
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const float2 t = fadd2(fadd2(leaf(a, 0), leaf(a, 2)), fadd2(leaf(a, 1), leaf(a, 3)));
            p[a] = fadd(t.x, t.y);
        }
    };
    partials([&](int a, int k) { return make_float2(x[a][2 * k], x[a][2 * k + 1]); });
    const float mu_own = __fmaf_rn(warp_rows8(p, lane, FAdd()), INV_N, nz);
    float mu[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) mu[a] = __shfl_sync(kFull, mu_own, 4 * a);
    partials([&](int a, int k) {
        const float2 d = fsub2(make_float2(x[a][2 * k], x[a][2 * k + 1]), make_float2(mu[a], mu[a]));
        return ffma2(d, d, nz2);
    });
    const float sig = kv_sigma(warp_rows8(p, lane, FAdd()), INV_N);
    if constexpr (APPLY) {
        const float inv_own = fdiv(1.0f, sig);
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const float inv = __shfl_sync(kFull, inv_own, 4 * a);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 v = ffma2(make_float2(x[a][2 * k], x[a][2 * k + 1]), make_float2(inv, inv), nz2);
                x[a][2 * k] = v.x;
                x[a][2 * k + 1] = v.y;
            }
        }
        if ((lane & 3) == 0) {
            const int t = warp + 16 * (lane >> 2);
            r[t] = fmul(r[t], sig);
        }
    }
    return fabsf(fsub(sig, 1.0f));
}

// A column pass (n = 128: column /= sigma, the column scale c[j] *= sigma). Column positions
// t = w + 16 a: the thread's levels pair a with a + 4 (stride 64), a + 2 (32), a + 1 (16); the
// warps' partials go to part [16][256] and thread j < 256 finishes column j's tree over the
// warps (strides 8 .. 1). mu_s, inv_s: [256] of shared memory. Returns |sigma - 1| of column
// threadIdx.x (threads < 256; 0 for the others). Four barriers: the first publishes the
// partials, the last the inverses; a column pass's reads of part, mu_s and inv_s all come
// before the next column pass writes them again (past one or more of these barriers).
__device__ __forceinline__ float kv_col_pass(float (&x)[8][8], float* c, float* part, float* mu_s, float* inv_s,
                                             int warp, int lane, float nz) {
    constexpr float INV_N = 1.0f / 128.0f;
    const int tid = threadIdx.x;
    const float2 nz2 = make_float2(nz, nz);
    // leaf(a, k): the leaves of columns 2k and 2k + 1 of row a as a pair, the two columns'
    // trees side by side
    auto partials = [&](auto leaf) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 s[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) s[a] = fadd2(leaf(a, k), leaf(a + 4, k));
            const float2 t = fadd2(fadd2(s[0], s[2]), fadd2(s[1], s[3]));
            part[warp * 256 + lane + 32 * (2 * k)] = t.x;
            part[warp * 256 + lane + 32 * (2 * k + 1)] = t.y;
        }
    };
    auto column_total = [&]() {
        float s[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) s[w] = fadd(part[w * 256 + tid], part[(w + 8) * 256 + tid]);
#pragma unroll
        for (int w = 0; w < 4; ++w) s[w] = fadd(s[w], s[w + 4]);
        return fadd(fadd(s[0], s[2]), fadd(s[1], s[3]));
    };
    partials([&](int a, int k) { return make_float2(x[a][2 * k], x[a][2 * k + 1]); });
    __syncthreads();
    if (tid < 256) mu_s[tid] = fmul(column_total(), INV_N);
    __syncthreads();
    float mu[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) mu[b] = mu_s[lane + 32 * b];
    partials([&](int a, int k) {
        const float2 d = fsub2(make_float2(x[a][2 * k], x[a][2 * k + 1]), make_float2(mu[2 * k], mu[2 * k + 1]));
        return ffma2(d, d, nz2);
    });
    __syncthreads();
    float dev = 0.f;
    if (tid < 256) {
        const float sig = kv_sigma(column_total(), INV_N);
        dev = fabsf(fsub(sig, 1.0f));
        inv_s[tid] = fdiv(1.0f, sig);
        c[tid] = fmul(c[tid], sig);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 inv = make_float2(inv_s[lane + 64 * k], inv_s[lane + 64 * k + 32]);
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const float2 v = ffma2(make_float2(x[a][2 * k], x[a][2 * k + 1]), inv, nz2);
            x[a][2 * k] = v.x;
            x[a][2 * k + 1] = v.y;
        }
    }
    return dev;
}

// Block maximum of v (non-negative) into *out, every thread calling; wmax: 16 floats of shared
// memory that no other block reduction uses until the next __syncthreads after this call.
__device__ __forceinline__ void block_max_to(float v, float* wmax, float* out) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = wmax[0];
        for (int i = 1; i < kKvWarps; ++i) m = fmaxf(m, wmax[i]);
        *out = m;
    }
}

// The codes of a tile in shared memory, one byte each, in the record's row order: K [128
// tokens][kCodeK bytes], V [256 channels][kCodeV bytes]; the padding word puts consecutive
// rows one bank apart.
constexpr int kCodeK = 260;
constexpr int kCodeV = 132;
constexpr int kCodeBytes = 256 * kCodeV;     // >= 128 kCodeK, and >= the 16 KB of column partials
constexpr int kTileBytes = 128 * 256 * 4;    // the fp32 copy of the unbalanced tile

// One code plane of width WK (kvarn_planes) from the codes of a tile, rows of NCOLS codes (K
// 256, V 128) STRIDE bytes apart: byte i of the plane packs 8 / WK codes of one row, code m at
// bits WK m, each code's bits sh .. sh + WK - 1; so 32-bit word i holds 32 / WK consecutive
// codes of one row at bits WK m. A thread forms a word from the 32-bit words of its codes: the
// fields of 4 bytes (each < 2^WK after the shift and mask) are squeezed together by shifts.
template <int WK, int NCOLS, int STRIDE>
__device__ __forceinline__ void kv_plane(uint32_t* plane, const uint8_t* codes, int sh) {
    constexpr int ROW_WORDS = NCOLS * WK / 32, PER_WORD = 32 / WK, NW = 8 / WK;
    constexpr uint32_t MASK = ((1u << WK) - 1u) * 0x01010101u;
    for (int i = threadIdx.x; i < 1024 * WK; i += kKvThreads) {
        const int row = i / ROW_WORDS, e0 = (i % ROW_WORDS) * PER_WORD;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(codes + row * STRIDE + e0);
        uint32_t out = 0;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            uint32_t t = (src[k] >> sh) & MASK;
            if constexpr (WK == 4) {
                t = (t | (t >> 4)) & 0x00FF00FFu;
                t = (t | (t >> 8)) & 0x0000FFFFu;
            } else if constexpr (WK == 2) {
                t = (t | (t >> 6)) & 0x000F000Fu;
                t = (t | (t >> 12)) & 0x000000FFu;
            } else if constexpr (WK == 1) {
                t = (t | (t >> 7)) & 0x00030003u;
                t = (t | (t >> 14)) & 0x0000000Fu;
            }
            out |= t << (4 * WK * k);
        }
        plane[i] = out;
    }
}

// grid (groups, H, 2 * D/256), 512 threads. Dynamic shared memory: the column partials
// [16][256] fp32, then (once the passes are done, over them) the codes; after them the staged
// rows of the half (tq6_0: [128][192] codes + [128][D/128] scales; 16-bit: [128][512]), then
// (once decoded, over them) the fp32 copy of the unbalanced tile.
// BITS: 0 = any code width and balancing read from the layout; 4 = 4-bit keys and values with
// the 16-pass balancing (an instance with only that code: fewer instruction-cache misses).
template <int JK, int BITS>
__global__ void __launch_bounds__(kKvThreads) seal_kvarn_kernel(Layout L, SealParams p, float nz) {
    constexpr int ROW = KvStage<JK>::ROW;
    const SealTaskPos tk = seal_task(p, blockIdx.x);
    const int nh = L.D / 256;
    const int h = blockIdx.y, w = blockIdx.z / nh, half = blockIdx.z % nh;
    const int fmt = L.fmt[w];
    const int bits = BITS ? BITS : kvarn_bits(fmt);
    const float Q = (float)((1 << bits) - 1);
    const int64_t unit = L.unit(tk.layer, tk.slot, h);
    extern __shared__ __align__(16) uint8_t kv_sm[];
    float* part = reinterpret_cast<float*>(kv_sm);                   // [16][256] column partials
    uint8_t* codes = kv_sm;                                          // codes, over part
    uint8_t* st = kv_sm + kCodeBytes;                                // staged rows
    uint16_t* sc = reinterpret_cast<uint16_t*>(st + 128 * ROW);      // tq6_0 scales [128][D/128]
    __shared__ float r[128], c[256], invS[128], Zs[128], invC[256], mu_s[256], inv_s[256];
    __shared__ uint16_t S16[128], Z16[128], C16[256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsc = L.D / 128;

    // stage the half's 128 journal rows (contiguous slots)
    {
        const int s0 = journal_slot(L, tk.pos0);
        if constexpr (JK == J_IN) {
            const int64_t row0 = p.seq[tk.b].src_row + (tk.pos0 - p.seq[tk.b].first_pos);
            const uint8_t* src = reinterpret_cast<const uint8_t*>((w ? p.v_src : p.k_src) + (row0 * L.H + h) * L.D) +
                                 512 * half;
            const int64_t rs = 2LL * L.H * L.D;
            for (int ci = threadIdx.x; ci < 128 * 32; ci += kKvThreads) {
                const int rr = ci >> 5, k = ci & 31;
                cp_async16(st + rr * ROW + 16 * k, src + rr * rs + 16 * k);
            }
        } else if constexpr (JK == J_TQ6) {
            const uint8_t* src = jcode_row(L, p.pool, w, unit, s0) + 192 * half;
            const int64_t jr = L.jrow_bytes;
            for (int ci = threadIdx.x; ci < 128 * 12; ci += kKvThreads) {
                const int rr = ci / 12, k = ci - 12 * rr;
                cp_async16(st + rr * ROW + 16 * k, src + rr * jr + 16 * k);
            }
            const uint8_t* ss = reinterpret_cast<const uint8_t*>(jscale_row(L, p.pool, w, unit, s0));
            for (int ci = threadIdx.x; ci < L.D / 8; ci += kKvThreads)
                cp_async16(reinterpret_cast<uint8_t*>(sc) + 16 * ci, ss + 16 * ci);
        } else {
            const uint8_t* src = reinterpret_cast<const uint8_t*>(jexact_row(L, p.pool, w, unit, s0)) + 512 * half;
            const int64_t rs = 2LL * L.D;
            for (int ci = threadIdx.x; ci < 128 * 32; ci += kKvThreads) {
                const int rr = ci >> 5, k = ci & 31;
                cp_async16(st + rr * ROW + 16 * k, src + rr * rs + 16 * k);
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
    }
    // the thread's part of the tile from the staged rows (x[a][b] = row warp + 16 a, channel
    // lane + 32 b), unit scales; the first barrier makes every thread's staged rows (cp.async,
    // each thread waited only for its own copies) visible to all. Once every thread has decoded
    // its values, a copy of them (x0: 16 float4 per thread, thread-major so a warp's accesses
    // are contiguous) replaces the staged rows: the codes and a second balancing read it.
    float x[8][8];
    float4* x0 = reinterpret_cast<float4*>(st);
    auto unit_scales = [&]() {
        for (int j = threadIdx.x; j < 256; j += kKvThreads) c[j] = 1.f;
        if (threadIdx.x < 128) r[threadIdx.x] = 1.f;
    };
    auto reload = [&]() {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const float4 v = x0[n * kKvThreads + threadIdx.x];
            x[n >> 1][4 * (n & 1)] = v.x;
            x[n >> 1][4 * (n & 1) + 1] = v.y;
            x[n >> 1][4 * (n & 1) + 2] = v.z;
            x[n >> 1][4 * (n & 1) + 3] = v.w;
        }
    };
    unit_scales();
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 8; ++a) kv_row<JK>(st, sc, warp + 16 * a, nsc, half, lane, x[a], L.journal, nz);
    __syncthreads();
#pragma unroll
    for (int n = 0; n < 16; ++n)
        x0[n * kKvThreads + threadIdx.x] = make_float4(x[n >> 1][4 * (n & 1)], x[n >> 1][4 * (n & 1) + 1],
                                                       x[n >> 1][4 * (n & 1) + 2], x[n >> 1][4 * (n & 1) + 3]);

    int passes = 16;
    if (BITS == 0 && L.kvarn_best) {
        // the KVarN reference configuration: 8 passes, keeping the state with the smallest
        // imbalance (largest |sigma - 1| over the lines the last pass left unbalanced). Pass p
        // measures the state of pass p - 1 on its own axis while it balances it; a measuring
        // row pass after pass 7 takes the last state's. Then the tile is balanced again from
        // the staged rows up to the kept pass (the same operations, so the same state).
        __shared__ float s_wmax[kKvWarps], s_eps[8];
        __shared__ int s_best;
        for (int pass = 0; pass < 8; ++pass) {
            const float dev = (pass & 1) == 0 ? kv_row_pass(x, r, warp, lane, nz)
                                              : kv_col_pass(x, c, part, mu_s, inv_s, warp, lane, nz);
            if (pass > 0) {
                block_max_to(dev, s_wmax, &s_eps[pass - 1]);
                __syncthreads();
            }
        }
        block_max_to(kv_row_pass<false>(x, r, warp, lane, nz), s_wmax, &s_eps[7]);
        if (threadIdx.x == 0) {
            int b = 0;
            for (int i = 1; i < 8; ++i)
                if (s_eps[i] < s_eps[b]) b = i;
            s_best = b;
        }
        __syncthreads();
        passes = s_best + 1;
        unit_scales();
        __syncthreads();
        reload();
    }
#pragma unroll 1
    for (int pass = 0; pass < passes; ++pass) {
        if ((pass & 1) == 0) kv_row_pass(x, r, warp, lane, nz);
        else kv_col_pass(x, c, part, mu_s, inv_s, warp, lane, nz);
    }

    // row rounding parameters: each row's extremes over the balanced values; lanes 4k .. 4k + 3
    // hold those of row warp + 16 k, whose row scale the same lane 4k updated
    {
        float lo8[8], hi8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            lo8[a] = 3.4e38f;
            hi8[a] = -3.4e38f;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                lo8[a] = fminf(lo8[a], x[a][b]);
                hi8[a] = fmaxf(hi8[a], x[a][b]);
            }
        }
        const float lo = warp_rows8(lo8, lane, FMin()), hi = warp_rows8(hi8, lane, FMax());
        if ((lane & 3) == 0) {
            const int t = warp + 16 * (lane >> 2);
            const uint16_t s16 = f2h_bits(fdiv(fmul(r[t], fsub(hi, lo)), Q));
            const uint16_t z16 = f2h_bits(fmul(r[t], lo));
            S16[t] = s16;
            Z16[t] = z16;
            const float sv = h2f(s16);
            invS[t] = (sv == 0.f) ? 0.f : fdiv(1.0f, sv);
            Zs[t] = h2f(z16);
            flag_nonfinite(L, p.pool, sv);
            flag_nonfinite(L, p.pool, Zs[t]);
        }
    }
    for (int j = threadIdx.x; j < 256; j += kKvThreads) {
        const uint16_t c16 = f2h_bits(c[j]);
        C16[j] = c16;
        invC[j] = fdiv(1.0f, h2f(c16));
        flag_nonfinite(L, p.pool, h2f(c16));
    }
    __syncthreads();

    // codes from the unbalanced values (x0) and the stored scales, laid out as the record's
    // rows: K token-major [128][kCodeK], V channel-major [256][kCodeV] (a warp's 32 channels of
    // one token then fall in 32 banks)
    reload();
    {
        float ic[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) ic[b] = invC[lane + 32 * b];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const int t = warp + 16 * a;
            const float is = invS[t], z = Zs[t];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int j = lane + 32 * b;
                float q = 0.f;
                if (is != 0.f) {
                    q = rintf(fmul(fsub(fmul(x[a][b], ic[b]), z), is));
                    q = fminf(fmaxf(q, 0.f), Q);
                }
                if (w == 0) codes[t * kCodeK + j] = (uint8_t)q;
                else codes[j * kCodeV + t] = (uint8_t)q;
            }
        }
    }
    __syncthreads();

    uint8_t* rec = body_rec(L, p.pool, w, unit, tk.g) + (int64_t)half * (4096 * bits + 1152);
    // code planes (kvarn_planes), 32-bit words at a time
    {
        int pw[2];
        const int np = kvarn_planes(bits, pw);
        uint32_t* plane = reinterpret_cast<uint32_t*>(rec);
        int sh = 0;
        for (int k = 0; k < np; ++k) {
            if (w == 0) {
                switch (pw[k]) {
                    case 1: kv_plane<1, 256, kCodeK>(plane, codes, sh); break;
                    case 2: kv_plane<2, 256, kCodeK>(plane, codes, sh); break;
                    case 4: kv_plane<4, 256, kCodeK>(plane, codes, sh); break;
                    default: kv_plane<8, 256, kCodeK>(plane, codes, sh); break;
                }
            } else {
                switch (pw[k]) {
                    case 1: kv_plane<1, 128, kCodeV>(plane, codes, sh); break;
                    case 2: kv_plane<2, 128, kCodeV>(plane, codes, sh); break;
                    case 4: kv_plane<4, 128, kCodeV>(plane, codes, sh); break;
                    default: kv_plane<8, 128, kCodeV>(plane, codes, sh); break;
                }
            }
            plane += 1024 * pw[k];
            sh += pw[k];
        }
    }
    uint16_t* sb = reinterpret_cast<uint16_t*>(rec + 4096 * bits);
    for (int i = threadIdx.x; i < 576; i += kKvThreads) {
        uint16_t x = 0;
        if (i < 128) x = S16[i];
        else if (i < 256) x = Z16[i - 128];
        else if (i < 512) x = C16[i - 256];
        sb[i] = x;
    }
}

template <int JK, int BITS>
int launch_kvarn_b(const Layout& L, const SealParams& p, int groups, cudaStream_t s) {
    constexpr int ROW = KvStage<JK>::ROW;
    const size_t stage = 128 * ROW + (JK == J_TQ6 ? 2 * L.D : 0);
    const size_t smem = kCodeBytes + (stage > kTileBytes ? stage : kTileBytes);
    auto fn = seal_kvarn_kernel<JK, BITS>;
    int e = (int)cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e) return e;
    dim3 grid(groups, L.H, 2 * (L.D / 256));
    fn<<<grid, kKvThreads, smem, s>>>(L, p, -0.0f);   // nz: see kv_row_pass
    return (int)cudaGetLastError();
}
template <int JK>
int launch_kvarn(const Layout& L, const SealParams& p, int groups, cudaStream_t s) {
    if (L.fmt[0] == KVQ_KVARN4 && L.fmt[1] == KVQ_KVARN4 && !L.kvarn_best) return launch_kvarn_b<JK, 4>(L, p, groups, s);
    return launch_kvarn_b<JK, 0>(L, p, groups, s);
}

}  // namespace

int launch_seal(const Layout& L, const SealParams& p, void* stream) {
    const int groups = p.n_layers * p.groups_per_layer;
    if (groups == 0) return 0;
    if (kvarn_bits(L.fmt[0])) {
        if (L.D % 256) return (int)cudaErrorInvalidValue;
        cudaStream_t s = (cudaStream_t)stream;
        if (p.k_src != nullptr) return launch_kvarn<J_IN>(L, p, groups, s);
        if (L.journal == KVQ_TQ6_0) return launch_kvarn<J_TQ6>(L, p, groups, s);
        if (L.journal == KVQ_BF16) return launch_kvarn<J_BF16>(L, p, groups, s);
        return launch_kvarn<J_F16>(L, p, groups, s);
    }
    return launch_seal_rows(L, p, stream);
}

int launch_seal_rows(const Layout& L, const SealParams& p, void* stream) {
    const int groups = p.n_layers * p.groups_per_layer;
    if (groups == 0) return 0;
    if (L.D % 128) return (int)cudaErrorInvalidValue;
    const int n_tiles = groups * L.H * 2 * (L.D / 128);
    cudaStream_t s = (cudaStream_t)stream;
    const bool tbq = (rotation_of(L.fmt[0]) == ROT_TBQ128);
    if (tbq != (rotation_of(L.fmt[1]) == ROT_TBQ128)) return (int)cudaErrorInvalidValue;   // one rotation per layout
    if (tbq) {
        if (L.fmt[0] == KVQ_TBQ4 && L.fmt[1] == KVQ_TBQ4) return launch_family<F_TBQ4_ONLY>(L, p, n_tiles, s);
        return launch_family<F_TBQ4>(L, p, n_tiles, s);
    }
    auto q84 = [](int f) { return f == KVQ_Q8_0 || f == KVQ_Q4_0; };
    if (q84(L.fmt[0]) && q84(L.fmt[1])) return launch_family<F_Q84>(L, p, n_tiles, s);
    return launch_family<F_Q>(L, p, n_tiles, s);
}

int query_sm_count(int device) {
    static int cached[64] = {0};
    if (device < 0 || device >= 64) return 1;
    if (cached[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) return 1;
        cached[device] = n;
    }
    return cached[device];
}

int upload_tables_seal(const FormatTables& t) {
    return (int)cudaMemcpyToSymbol(c_tab, &t, sizeof(FormatTables));
}

}  // namespace kvq
