// Split-K decode attention over every region of the cache, then a log-sum-exp merge.
//
// Work item = (sequence, KV head, span of positions inside one region). Each CTA of
// decode_split_kernel streams its span in tiles: all threads decode the tile's K and V
// records into shared memory as fp16 (scales applied), then warps run tensor-core
// mma.sync m16n8k16 (fp16 in, fp32 accumulate): S^T = K Q^T with positions on M and the
// GQA query group on N, an online softmax in the log2 domain, and O^T += V^T P^T with
// channels on M. Rotated regions (body, tq6_0 ring span) are read with the rotated query
// R q; at the end of the item the partial output is rotated back (R^T), so every partial
// is in the original domain (KV cache math, "rotate first": the query is rotated once and
// the output rotated back once; R^T distributes over the merge sum).
// decode_merge_kernel combines the partials of one (sequence, KV head) under one softmax:
// m* = max m_c, l* = sum 2^(m_c - m*) l_c, o = sum 2^(m_c - m*) o_c / l* (KV Cache
// Precision Tail §2: results combined under one softmax; HAL #582 §5 P2: exact online-
// softmax combine of typed regions).
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cfloat>
#include <mutex>
#include "device_common.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTbqScale = 0.0883883461356163f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void store8(__half* dst, const float (&v)[8]) {
    uint4 u;
    u.x = pack_h2(v[0], v[1]);
    u.y = pack_h2(v[2], v[3]);
    u.z = pack_h2(v[4], v[5]);
    u.w = pack_h2(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = u;
}
// 8 values as fp16 (dst) and, with lo, the fp16 remainders v - fp16(v) (lo): hi + lo carries
// 22 significant bits of each value.
__device__ __forceinline__ void store8_split(__half* dst, __half* lo, const float (&v)[8]) {
    if (!lo) {
        store8(dst, v);
        return;
    }
    float h[8], r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        h[k] = __half2float(__float2half_rn(v[k]));
        r[k] = v[k] - h[k];
    }
    store8(dst, h);
    store8(lo, r);
}

// Block-wide FWHT over rows of n values (shared fp32), ascending strides.
__device__ void block_fwht_rows(float* xs, int total, int n) {
    for (int s = 1; s < n; s <<= 1) {
        for (int p = threadIdx.x; p < total / 2; p += blockDim.x) {
            const int blk = p / (n / 2), q = p % (n / 2);
            const int i = blk * n + (q / s) * 2 * s + (q % s);
            const float a = xs[i], b = xs[i + s];
            xs[i] = a + b;
            xs[i + s] = a - b;
        }
        __syncthreads();
    }
}

// Forward (inverse = false) or inverse rotation of `rows` vectors of D values in xs.
__device__ void rotate_rows(float* xs, int rows, int D, int rot, bool inverse) {
    const int total = rows * D;
    if (rot == ROT_HAD256) {
        block_fwht_rows(xs, total, 256);
        for (int i = threadIdx.x; i < total; i += blockDim.x) xs[i] *= 0.0625f;
        __syncthreads();
    } else if (rot == ROT_TBQ128) {
        const int first = inverse ? 1 : 0;
        for (int i = threadIdx.x; i < total; i += blockDim.x)
            if (sign_neg(first, i & 127)) xs[i] = -xs[i];
        __syncthreads();
        block_fwht_rows(xs, total, 128);
        for (int i = threadIdx.x; i < total; i += blockDim.x) {
            float y = xs[i];
            if (sign_neg(1 - first, i & 127)) y = -y;
            xs[i] = y * kTbqScale;
        }
        __syncthreads();
    }
}

struct Item {
    int b, h, kind, t0, t1, slot;
};

__device__ __forceinline__ Item decode_item(const AttnParams& p, int item) {
    Item it;
    int b = 0;
    while (b + 1 < p.n_seq && p.seq[b + 1].first_item <= item) ++b;
    const SeqSpan& s = p.seq[b];
    const int local = item - s.first_item;
    it.b = b;
    it.h = local / s.items_per_head;
    int c = local % s.items_per_head;
    int r = 0;
    while (r < 3 && c >= s.nchunk[r]) { c -= s.nchunk[r]; ++r; }
    it.kind = s.kind[r];
    const int ck = (it.kind == RK_RING) ? p.ring_chunk : p.chunk;
    it.t0 = s.lo[r] + c * ck;
    it.t1 = min(it.t0 + ck, s.hi[r]);
    it.slot = s.slot;
    return it;
}

// --------------------------------------------------------------------------- tile fill
// Each fill first issues every global load of its share of the tile into registers, then
// decodes and stores to shared memory, so a thread has all its loads in flight at once.
// Token-major exact rows (sink, exact tail, exact journal) into dst[TILE][LD].
template <int D, int TILE, int LD>
__device__ void fill_exact(const Layout& L, const void* pool, int w, int64_t unit, int kind, int tstart,
                           int nvalid, __half* dst) {
    constexpr int U = D / 8;     // 16-byte units per row
    constexpr int IT = (TILE * U + kThreads - 1) / kThreads;
    const int fmt = (kind == RK_SINK) ? KVQ_F16 : (kind == RK_TAIL ? L.tail_fmt : L.journal);
    uint4 raw[IT];
#pragma unroll
    for (int k = 0; k < IT; ++k) {
        const int e = threadIdx.x + k * kThreads;
        const int i = e / U, u = e % U;
        raw[k] = make_uint4(0, 0, 0, 0);
        if (e < TILE * U && i < nvalid) {
            const int pos = tstart + i;
            const uint16_t* row;
            if (kind == RK_SINK) row = sink_row(L, pool, w, unit, pos);
            else if (kind == RK_TAIL) row = tail_row(L, pool, w, unit, pos % L.T);
            else row = jexact_row(L, pool, w, unit, journal_slot(L, pos));
            raw[k] = __ldg(reinterpret_cast<const uint4*>(row + 8 * u));
        }
    }
#pragma unroll
    for (int k = 0; k < IT; ++k) {
        const int e = threadIdx.x + k * kThreads;
        if (e >= TILE * U) break;
        const int i = e / U, u = e % U;
        __half* o = dst + i * LD + 8 * u;
        if (fmt == KVQ_F16 || i >= nvalid) {
            *reinterpret_cast<uint4*>(o) = raw[k];
        } else {
            const uint16_t* r16 = reinterpret_cast<const uint16_t*>(&raw[k]);
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = bf2f(r16[j]);
            store8(o, v);
        }
    }
}

// tq6_0 ring rows (rotated domain), token-major.
template <int D, int TILE, int LD>
__device__ void fill_ring(const Layout& L, const void* pool, int w, int64_t unit, int tstart, int nvalid,
                          __half* dst) {
    constexpr int U = D / 8;
    constexpr int IT = (TILE * U + kThreads - 1) / kThreads;
    uint32_t ql[IT];
    uint16_t qh[IT], ds[IT];
#pragma unroll
    for (int k = 0; k < IT; ++k) {
        const int e = threadIdx.x + k * kThreads;
        const int i = e / U, u = e % U;
        ql[k] = 0; qh[k] = 0; ds[k] = 0;
        if (e < TILE * U && i < nvalid) {
            const int slot = journal_slot(L, tstart + i);
            const int c0 = 8 * u, blk = c0 >> 7, j0 = c0 & 127;
            const uint8_t* row = jcode_row(L, pool, w, unit, slot) + 96 * blk;
            ql[k] = __ldg(reinterpret_cast<const uint32_t*>(row + (j0 >> 1)));
            qh[k] = __ldg(reinterpret_cast<const uint16_t*>(row + 64 + (j0 >> 2)));
            ds[k] = __ldg(jscale_row(L, pool, w, unit, slot) + blk);
        }
    }
#pragma unroll
    for (int k = 0; k < IT; ++k) {
        const int e = threadIdx.x + k * kThreads;
        if (e >= TILE * U) break;
        const int i = e / U, u = e % U;
        __half* o = dst + i * LD + 8 * u;
        const float d = h2f(ds[k]);
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int code = ((ql[k] >> (4 * j)) & 15) | (((qh[k] >> (2 * j)) & 3) << 4);
            v[j] = (i < nvalid) ? (float)(code - 32) * d : 0.f;
        }
        store8(o, v);
    }
}

// Codes e0 .. e0 + 7 (e0 a multiple of 8) of row `row` of a KVarN tile's code planes (rows of
// len codes; see kvarn_planes): each plane's 8 codes are w consecutive bytes, one aligned load.
__device__ __forceinline__ uint64_t load_wbytes(const uint8_t* p, int w) {
    switch (w) {
        case 1: return *p;
        case 2: return *reinterpret_cast<const uint16_t*>(p);
        case 4: return *reinterpret_cast<const uint32_t*>(p);
        default: return *reinterpret_cast<const uint64_t*>(p);
    }
}
__device__ __forceinline__ void kvarn_codes8(const uint8_t* tile, int bits, int len, int row, int e0, int (&code)[8]) {
    const int w0 = bits >= 4 ? (bits == 8 ? 8 : 4) : 2, w1 = bits - w0;
    const int64_t at = (int64_t)row * len + e0;
    const uint64_t a = load_wbytes(tile + at * w0 / 8, w0);
    const uint64_t b = w1 ? load_wbytes(tile + 4096 * w0 + at * w1 / 8, w1) : 0;
#pragma unroll
    for (int m = 0; m < 8; ++m)
        code[m] = (int)(((a >> (w0 * m)) & ((1u << w0) - 1)) | (((b >> (w1 * m)) & ((1u << w1) - 1)) << w0));
}

// Value of channel c of row t (token-major) of a Q5_0 / Q6_0 / Q4_1 / Q5_1 record.
__device__ __forceinline__ float qblock_value(const uint8_t* rec, int fmt, int D, int t, int c) {
    const int bits = qblock_bits(fmt);
    int code = (rec[t * (D / 2) + (c >> 1)] >> ((c & 1) * 4)) & 15;
    if (bits == 5) code |= ((rec[64 * D + t * (D / 8) + (c >> 3)] >> (c & 7)) & 1) << 4;
    else if (bits == 6) code |= ((rec[64 * D + t * (D / 4) + (c >> 2)] >> (2 * (c & 3))) & 3) << 4;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(rec + record_code_bytes(fmt, D));
    const float d = h2f(sc[t * (D / 32) + (c >> 5)]);
    const int L = qblock_sym_levels(fmt);
    if (L) return (float)(code - (L + 1)) * d;
    return (float)code * d + h2f(sc[4 * D + t * (D / 32) + (c >> 5)]);
}

// Value of channel c of row t (token-major) of a turbo3 or tq5_0 record (rotated domain).
__device__ __forceinline__ float rot_block_value(const uint8_t* rec, int fmt, int D, int t, int c) {
    if (fmt == KVQ_TURBO3) {
        const int code = ((rec[t * (D / 4) + (c >> 2)] >> (2 * (c & 3))) & 3) |
                         (((rec[32 * D + t * (D / 8) + (c >> 3)] >> (c & 7)) & 1) << 2);
        return c_tab.cent3[code] * h2f(reinterpret_cast<const uint16_t*>(rec + 48 * D)[t * (D / 128) + (c >> 7)]);
    }
    const int code = ((rec[t * (D / 2) + (c >> 1)] >> ((c & 1) * 4)) & 15) |
                     (((rec[64 * D + t * (D / 8) + (c >> 3)] >> (c & 7)) & 1) << 4);
    return (float)(code - 16) * h2f(reinterpret_cast<const uint16_t*>(rec + 80 * D)[t * (D / 128) + (c >> 7)]);
}

// Channels c0 .. c0 + 7 (c0 a multiple of 8) of row t of a token-major Q5_0 / Q6_0 / Q4_1 /
// Q5_1 / turbo3 / tq5_0 record: one load per plane and one per scale for the 8 values.
__device__ __forceinline__ void tok_values8(const uint8_t* rec, int fmt, int D, int t, int c0, float (&v)[8]) {
    if (fmt == KVQ_TURBO3) {
        const uint32_t lo = *reinterpret_cast<const uint16_t*>(rec + t * (D / 4) + (c0 >> 2));   // 2 bits each
        const uint32_t hb = rec[32 * D + t * (D / 8) + (c0 >> 3)];                             // bit 2
        const float n = h2f(reinterpret_cast<const uint16_t*>(rec + 48 * D)[t * (D / 128) + (c0 >> 7)]);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = c_tab.cent3[((lo >> (2 * k)) & 3) | (((hb >> k) & 1) << 2)] * n;
        return;
    }
    const uint32_t w4 = *reinterpret_cast<const uint32_t*>(rec + t * (D / 2) + (c0 >> 1));    // nibbles
    const int bits = fmt == KVQ_TQ5_0 ? 5 : qblock_bits(fmt);
    uint32_t hb = 0;
    if (bits == 5) hb = rec[64 * D + t * (D / 8) + (c0 >> 3)];
    else if (bits == 6) hb = *reinterpret_cast<const uint16_t*>(rec + 64 * D + t * (D / 4) + (c0 >> 2));
    int code[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        code[k] = (int)((w4 >> (4 * k)) & 15);
        if (bits == 5) code[k] |= (int)((hb >> k) & 1) << 4;
        else if (bits == 6) code[k] |= (int)((hb >> (2 * k)) & 3) << 4;
    }
    if (fmt == KVQ_TQ5_0) {
        const float d = h2f(reinterpret_cast<const uint16_t*>(rec + 80 * D)[t * (D / 128) + (c0 >> 7)]);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = (float)(code[k] - 16) * d;
        return;
    }
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(rec + record_code_bytes(fmt, D));
    const float d = h2f(sc[t * (D / 32) + (c0 >> 5)]);
    const int L = qblock_sym_levels(fmt);
    if (L) {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = (float)(code[k] - (L + 1)) * d;
    } else {
        const float m = h2f(sc[4 * D + t * (D / 32) + (c0 >> 5)]);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = (float)code[k] * d + m;
    }
}

// Body K records (token-major) of one tile: positions [tstart, tstart + TILE) of group g.
template <int D, int TILE, int LD>
__device__ void fill_body_k(const Layout& L, const void* pool, int64_t unit, int g, int rel, __half* dst,
                            const float* cent, __half* lo) {
    const int fmt = L.fmt[0];
    const uint8_t* rec = body_rec(L, pool, 0, unit, g);
    constexpr int U = D / 8;
    for (int e = threadIdx.x; e < TILE * U; e += kThreads) {
        const int i = e / U, u = e % U;
        const int t = rel + i, c0 = 8 * u;
        float v[8];
        if (qblock_bits(fmt) || fmt == KVQ_TURBO3 || fmt == KVQ_TQ5_0) {
            tok_values8(rec, fmt, D, t, c0, v);
        } else if (fmt == KVQ_TBQ4) {
            const uint32_t w4 = *reinterpret_cast<const uint32_t*>(rec + t * (D / 2) + (c0 >> 1));
            const float n = h2f(reinterpret_cast<const uint16_t*>(rec + 64 * D)[t * (D / 128) + (c0 >> 7)]);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = cent[(w4 >> (4 * k)) & 15] * n;
        } else if (fmt == KVQ_Q8_0) {
            const uint2 w8 = *reinterpret_cast<const uint2*>(rec + t * D + c0);
            const float d = h2f(reinterpret_cast<const uint16_t*>(rec + 128 * D)[t * (D / 32) + (c0 >> 5)]);
            const int8_t* q = reinterpret_cast<const int8_t*>(&w8);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = (float)q[k] * d;
        } else if (fmt == KVQ_Q4_0) {
            const uint32_t w4 = *reinterpret_cast<const uint32_t*>(rec + t * (D / 2) + (c0 >> 1));
            const float d = h2f(reinterpret_cast<const uint16_t*>(rec + 64 * D)[t * (D / 32) + (c0 >> 5)]);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = (float)((int)((w4 >> (4 * k)) & 15) - 8) * d;
        } else {   // KVarN (any code width: kvarn_code reads the planes)
            const int bits = kvarn_bits(fmt);
            const int hh = c0 >> 8, j0 = c0 & 255;
            const uint8_t* tr = rec + (int64_t)hh * (4096 * bits + 1152);
            const uint16_t* sb = reinterpret_cast<const uint16_t*>(tr + 4096 * bits);
            const float S = h2f(sb[t]), Z = h2f(sb[128 + t]);
            int code[8];
            kvarn_codes8(tr, bits, 256, t, j0, code);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = ((float)code[k] * S + Z) * h2f(sb[256 + j0 + k]);
        }
        store8_split(dst + i * LD + c0, lo ? lo + i * LD + c0 : nullptr, v);
    }
}

// Body V records (channel-major) of one tile into dst[D][LDV] (channel-major smem).
template <int D, int TILE, int LDV>
__device__ void fill_body_v(const Layout& L, const void* pool, int64_t unit, int g, int rel, __half* dst,
                            const float* cent, __half* lo) {
    const int fmt = L.fmt[1];
    const uint8_t* rec = body_rec(L, pool, 1, unit, g);
    constexpr int U = TILE / 8;   // 8-token units per channel
    for (int e = threadIdx.x; e < D * U; e += kThreads) {
        const int c = e / U, u = e % U;
        const int t0 = rel + 8 * u;
        float v[8];
        if (qblock_bits(fmt)) {   // token-major V
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = qblock_value(rec, fmt, D, t0 + k, c);
        } else if (fmt == KVQ_TURBO3 || fmt == KVQ_TQ5_0) {   // token-major V
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = rot_block_value(rec, fmt, D, t0 + k, c);
        } else if (fmt == KVQ_TBQ4) {
            const uint32_t w4 = *reinterpret_cast<const uint32_t*>(rec + c * 64 + (t0 >> 1));
            const uint16_t* nr = reinterpret_cast<const uint16_t*>(rec + 64 * D);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = cent[(w4 >> (4 * k)) & 15] * h2f(nr[(t0 + k) * (D / 128) + (c >> 7)]);
        } else if (fmt == KVQ_Q4_0) {
            const uint32_t w4 = *reinterpret_cast<const uint32_t*>(rec + c * 64 + (t0 >> 1));
            const uint16_t* dr = reinterpret_cast<const uint16_t*>(rec + 64 * D);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = (float)((int)((w4 >> (4 * k)) & 15) - 8) * h2f(dr[(t0 + k) * (D / 32) + (c >> 5)]);
        } else if (fmt == KVQ_Q8_0) {
            const uint2 w8 = *reinterpret_cast<const uint2*>(rec + c * 128 + t0);
            const int8_t* q = reinterpret_cast<const int8_t*>(&w8);
            const uint16_t* dr = reinterpret_cast<const uint16_t*>(rec + 128 * D);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = (float)q[k] * h2f(dr[(t0 + k) * (D / 32) + (c >> 5)]);
        } else {   // KVarN (any code width)
            const int bits = kvarn_bits(fmt);
            const int hh = c >> 8, j = c & 255;
            const uint8_t* tr = rec + (int64_t)hh * (4096 * bits + 1152);
            const uint16_t* sb = reinterpret_cast<const uint16_t*>(tr + 4096 * bits);
            const float C = h2f(sb[256 + j]);
            int code[8];
            kvarn_codes8(tr, bits, 128, j, t0, code);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = ((float)code[k] * h2f(sb[t0 + k]) + h2f(sb[128 + t0 + k])) * C;
        }
        store8_split(dst + c * LDV + t0 - rel, lo ? lo + c * LDV + t0 - rel : nullptr, v);
    }
}

// --------------------------------------------------------------------------- split kernel
template <int D, int NQ>
struct Cfg {
    static constexpr int TILE = (D == 512) ? 32 : 64;
    static constexpr int LDK = D + 8;              // token-major row stride (halves)
    static constexpr int LDV = TILE + 8;           // channel-major row stride (halves)
    static constexpr int LDP = TILE + 8;
    static constexpr int K_BYTES = TILE * LDK * 2;
    static constexpr int V_BYTES = (TILE * LDK > D * LDV ? TILE * LDK : D * LDV) * 2;
    static constexpr int Q_BYTES = NQ * LDK * 2;
    static constexpr int S_BYTES = TILE * NQ * 4;
    static constexpr int P_BYTES = NQ * LDP * 2;
    static constexpr int QF_BYTES = NQ * D * 4;    // fp32 staging of q / the output rows
    static constexpr int SMEM = K_BYTES + V_BYTES + Q_BYTES + S_BYTES + P_BYTES + QF_BYTES + 64 * 4 + 16 * 4 +
                                K_BYTES + V_BYTES;   // the fp16 remainders of body K and V tiles
};

template <int D, int NQ>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(Layout L, AttnParams p) {
    using C = Cfg<D, NQ>;
    constexpr int TILE = C::TILE, LDK = C::LDK, LDV = C::LDV, LDP = C::LDP;
    extern __shared__ __align__(16) uint8_t smem[];
    __half* Ks = reinterpret_cast<__half*>(smem);
    __half* Vs = reinterpret_cast<__half*>(smem + C::K_BYTES);
    __half* Qs = reinterpret_cast<__half*>(smem + C::K_BYTES + C::V_BYTES);
    float* Ss = reinterpret_cast<float*>(smem + C::K_BYTES + C::V_BYTES + C::Q_BYTES);
    __half* Ps = reinterpret_cast<__half*>(smem + C::K_BYTES + C::V_BYTES + C::Q_BYTES + C::S_BYTES);
    float* QF = reinterpret_cast<float*>(smem + C::K_BYTES + C::V_BYTES + C::Q_BYTES + C::S_BYTES + C::P_BYTES);
    float* stat = QF + NQ * D;          // m[16], l[16], alpha[16], cent[16]
    float* m_run = stat;
    float* l_run = stat + 16;
    float* alpha = stat + 32;
    float* cent = stat + 48;
    __half* Ks_lo = reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(stat + 64 + 16));
    __half* Vs_lo = reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(Ks_lo) + C::K_BYTES);

    const Item it = decode_item(p, blockIdx.x);
    // body tiles of the 32-value block formats beyond Q8_0 / Q4_0 (and of turbo3, tq5_0) are held as fp16 values plus
    // fp16 remainders, and both go through the mma: an fp16 value of code x d (+ m) alone is too
    // coarse for the decode tolerance where the softmax is sharp
    auto split_fmt = [](int f) { return qblock_bits(f) != 0 || f == KVQ_TURBO3 || f == KVQ_TQ5_0; };
    const bool lo_now = it.kind == RK_BODY && (split_fmt(L.fmt[0]) || split_fmt(L.fmt[1]));
    const int G = L.G;
    const int64_t unit = L.unit(p.layer, it.slot, it.h);
    const bool rotated = (it.kind == RK_BODY || it.kind == RK_RING) && L.rot != ROT_NONE;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;

    if (threadIdx.x < 16) {
        m_run[threadIdx.x] = -INFINITY;
        l_run[threadIdx.x] = 0.f;
        cent[threadIdx.x] = c_tab.cent[threadIdx.x];
    }
    // query rows of this KV head, rotated when the item reads a rotated region
    const uint16_t* q = p.q + ((int64_t)it.b * L.Hq + (int64_t)it.h * G) * D;
    for (int e = threadIdx.x; e < NQ * D; e += kThreads) {
        const int r = e / D;
        QF[e] = (r < G) ? h2f(q[e]) : 0.f;
    }
    __syncthreads();
    if (rotated) rotate_rows(QF, NQ, D, L.rot, false);
    for (int e = threadIdx.x; e < NQ * D; e += kThreads) {
        const int r = e / D, c = e % D;
        Qs[r * LDK + c] = __float2half_rn(QF[e]);
    }
    const float sc = L.scale * kLog2e;
    const bool v_chmajor = (it.kind == RK_BODY);

    constexpr int MT = D / 128;          // PV m-tiles of 16 channels per warp (warp: D/8 channels)
    constexpr int NT = NQ / 8;
    float acc[MT][NT][4];
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int bq = 0; bq < NT; ++bq)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[a][bq][k] = 0.f;
    __syncthreads();

    for (int tstart = it.t0; tstart < it.t1; tstart += TILE) {
        const int nvalid = min(TILE, it.t1 - tstart);
        // ---- decode the tile into shared memory
        if (it.kind == RK_BODY) {
            const int g = (tstart - kSink) / kGroup, rel = (tstart - kSink) % kGroup;
            fill_body_k<D, TILE, LDK>(L, p.pool, unit, g, rel, Ks, cent, lo_now ? Ks_lo : nullptr);
            fill_body_v<D, TILE, LDV>(L, p.pool, unit, g, rel, Vs, cent, lo_now ? Vs_lo : nullptr);
        } else if (it.kind == RK_RING) {
            fill_ring<D, TILE, LDK>(L, p.pool, 0, unit, tstart, nvalid, Ks);
            fill_ring<D, TILE, LDK>(L, p.pool, 1, unit, tstart, nvalid, Vs);
        } else {
            fill_exact<D, TILE, LDK>(L, p.pool, 0, unit, it.kind, tstart, nvalid, Ks);
            fill_exact<D, TILE, LDK>(L, p.pool, 1, unit, it.kind, tstart, nvalid, Vs);
        }
        __syncthreads();
        // ---- scores: S^T[tok][q] = K Q^T, positions on M
        if (warp < TILE / 16) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t a0, a1, a2, a3, b0, b1;
                    ldsm_x4(smem_u32(Ks + (warp * 16 + (lane & 15)) * LDK + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
                    ldsm_x2(smem_u32(Qs + (nt * 8 + (lane & 7)) * LDK + ks * 16 + ((lane >> 3) & 1) * 8), b0, b1);
                    mma16816(c4, a0, a1, a2, a3, b0, b1);
                    if (lo_now) {
                        ldsm_x4(smem_u32(Ks_lo + (warp * 16 + (lane & 15)) * LDK + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
                        mma16816(c4, a0, a1, a2, a3, b0, b1);
                    }
                }
                const int r0 = warp * 16 + gq, qc = nt * 8 + 2 * tq;
                Ss[r0 * NQ + qc] = (r0 < nvalid) ? c4[0] * sc : -INFINITY;
                Ss[r0 * NQ + qc + 1] = (r0 < nvalid) ? c4[1] * sc : -INFINITY;
                Ss[(r0 + 8) * NQ + qc] = (r0 + 8 < nvalid) ? c4[2] * sc : -INFINITY;
                Ss[(r0 + 8) * NQ + qc + 1] = (r0 + 8 < nvalid) ? c4[3] * sc : -INFINITY;
            }
        }
        __syncthreads();
        // ---- online softmax (log2 domain), one warp per query
        for (int qi = warp; qi < NQ; qi += kThreads / 32) {
            float mt = -INFINITY;
            for (int t = lane; t < TILE; t += 32) mt = fmaxf(mt, Ss[t * NQ + qi]);
#pragma unroll
            for (int s = 16; s >= 1; s >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, s));
            const float mo = m_run[qi];
            const float mn = fmaxf(mo, mt);
            const float a = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
            float sum = 0.f;
            for (int t = lane; t < TILE; t += 32) {
                const float s = Ss[t * NQ + qi];
                const float pv = (mn == -INFINITY) ? 0.f : exp2f(s - mn);
                const __half ph = __float2half_rn(pv);
                Ps[qi * LDP + t] = ph;
                sum += __half2float(ph);
            }
#pragma unroll
            for (int s = 16; s >= 1; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
            __syncwarp();
            if (lane == 0) {
                m_run[qi] = mn;
                l_run[qi] = l_run[qi] * a + sum;
                alpha[qi] = a;
            }
        }
        __syncthreads();
        // ---- O^T[ch][q] += V^T P^T, channels on M; warp owns D/8 channels
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int ch0 = warp * (D / 8) + mt * 16;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float a0 = alpha[nt * 8 + 2 * tq], a1 = alpha[nt * 8 + 2 * tq + 1];
                acc[mt][nt][0] *= a0;
                acc[mt][nt][1] *= a1;
                acc[mt][nt][2] *= a0;
                acc[mt][nt][3] *= a1;
            }
#pragma unroll
            for (int ks = 0; ks < TILE / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                const int mi = lane >> 3, ri = lane & 7;
                if (v_chmajor) {
                    ldsm_x4(smem_u32(Vs + (ch0 + (mi & 1) * 8 + ri) * LDV + ks * 16 + (mi >> 1) * 8), a0, a1, a2, a3);
                } else {
                    ldsm_x4_t(smem_u32(Vs + (ks * 16 + (mi >> 1) * 8 + ri) * LDK + ch0 + (mi & 1) * 8), a0, a1, a2, a3);
                }
                uint32_t e0 = 0, e1 = 0, e2 = 0, e3 = 0;
                if (lo_now)   // body tiles are channel-major
                    ldsm_x4(smem_u32(Vs_lo + (ch0 + (mi & 1) * 8 + ri) * LDV + ks * 16 + (mi >> 1) * 8), e0, e1, e2, e3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    uint32_t b0, b1;
                    ldsm_x2(smem_u32(Ps + (nt * 8 + (lane & 7)) * LDP + ks * 16 + ((lane >> 3) & 1) * 8), b0, b1);
                    mma16816(acc[mt][nt], a0, a1, a2, a3, b0, b1);
                    if (lo_now) mma16816(acc[mt][nt], e0, e1, e2, e3, b0, b1);
                }
            }
        }
        __syncthreads();
    }

    // ---- partial: o in the original domain (rotated items rotated back), m and l
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int ch0 = warp * (D / 8) + mt * 16;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int qc = nt * 8 + 2 * tq;
            QF[qc * D + ch0 + gq] = acc[mt][nt][0];
            QF[(qc + 1) * D + ch0 + gq] = acc[mt][nt][1];
            QF[qc * D + ch0 + gq + 8] = acc[mt][nt][2];
            QF[(qc + 1) * D + ch0 + gq + 8] = acc[mt][nt][3];
        }
    }
    __syncthreads();
    if (rotated) rotate_rows(QF, NQ, D, L.rot, true);
    float* part = p.partials + (size_t)blockIdx.x * (2 * NQ + NQ * D);
    if (threadIdx.x < NQ) {
        part[threadIdx.x] = m_run[threadIdx.x];
        part[NQ + threadIdx.x] = l_run[threadIdx.x];
    }
    float4* po = reinterpret_cast<float4*>(part + 2 * NQ);
    const float4* qf4 = reinterpret_cast<const float4*>(QF);
    for (int e = threadIdx.x; e < NQ * D / 4; e += kThreads) po[e] = qf4[e];
}

// --------------------------------------------------------------------------- merge kernel
// grid (n_seq * H, D / 32); 256 threads. Phase 1: per query, the global max m* and
// l* = sum 2^(m_c - m*) l_c, and every partial's weight 2^(m_c - m*) into shared memory.
// Phase 2: thread (item slice, query, channel) sums w_c o_c over its slice of the partials
// with eight independent loads in flight; slices meet in shared memory.
constexpr int kMergeMaxItems = 1024;

// grid (n_seq * H, D / 8), 256 threads: block (bh, y) combines the partials of sequence
// bh / H, KV head bh % H for channels [8y, 8y + 8). Every partial's m and l are loaded at once
// (one thread per partial) into shared memory; a warp per query forms m*, the weights
// 2^(m_c - m*) and l*; then each thread issues the loads of all its partials' slices before
// accumulating them.
template <int D, int NQ>
__global__ void __launch_bounds__(256) decode_merge_kernel(Layout L, AttnParams p) {
    grid_dep_wait();          // the partials of the launch ahead are complete and visible
    // the next layer's decode kernel may start now: its items read nothing this kernel writes
    // and write their partials only after waiting for it (AttnParams::early)
    grid_dep_launch();
    const int bh = blockIdx.x;
    const int b = bh / L.H, h = bh % L.H;
    const SeqSpan& s = p.seq[b];
    const int first = s.first_item + h * s.items_per_head, cnt_r = s.items_per_head;
    const int bfirst = s.body_first + h * s.body_per_head;
    const int cnt = cnt_r + s.body_per_head;
    const int G = L.G;
    extern __shared__ float msm[];
    float* wgt = msm;                                   // [cnt][NQ]: m_c, then the weights
    float* lsm = msm + (size_t)cnt * NQ;                // [cnt][NQ]: l_c
    __shared__ float lstar[NQ];
    constexpr int FPI = 2 * NQ;                         // float4 slices per partial (8 channels x NQ)
    constexpr int IL = 256 / FPI;                       // partials in flight per pass
    __shared__ float4 red4[IL][FPI];
    auto item_of = [&](int c) { return c < cnt_r ? first + c : bfirst + (c - cnt_r); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t stride = 2 * NQ + NQ * D;
    // this thread's first U output slices are loaded now: they do not depend on the weights, so
    // their latency overlaps the round trip of m and l below
    const int c0 = blockIdx.y * 8;
    const int il = threadIdx.x / FPI, f = threadIdx.x % FPI;
    const int qi = f >> 1, half = f & 1;
    constexpr int U = 8;
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = il + IL * u;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (qi < G && c < cnt)
            v[u] = *reinterpret_cast<const float4*>(p.partials + item_of(c) * stride + 2 * NQ + qi * D + c0 + 4 * half);
    }
    for (int c = threadIdx.x; c < cnt; c += blockDim.x) {
        const float4* pc = reinterpret_cast<const float4*>(p.partials + item_of(c) * stride);
        float4 mv[NQ / 4], lv[NQ / 4];
#pragma unroll
        for (int k = 0; k < NQ / 4; ++k) {
            mv[k] = pc[k];
            lv[k] = pc[NQ / 4 + k];
        }
#pragma unroll
        for (int k = 0; k < NQ / 4; ++k) {
            reinterpret_cast<float4*>(wgt + c * NQ)[k] = mv[k];
            reinterpret_cast<float4*>(lsm + c * NQ)[k] = lv[k];
        }
    }
    __syncthreads();
    for (int qw = warp; qw < G; qw += 8) {
        float m = -INFINITY;
        for (int c = lane; c < cnt; c += 32) m = fmaxf(m, wgt[c * NQ + qw]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int c = lane; c < cnt; c += 32) {
            const float mc = wgt[c * NQ + qw];
            const float w = (mc == -INFINITY) ? 0.f : exp2f(mc - m);
            wgt[c * NQ + qw] = w;
            l += w * lsm[c * NQ + qw];
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) lstar[qw] = l;
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (qi < G) {
        for (int cb = il; cb < cnt; cb += IL * U) {
            if (cb != il) {   // slices past the first U (prefetched above)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = cb + IL * u;
                    v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (c < cnt)
                        v[u] = *reinterpret_cast<const float4*>(p.partials + item_of(c) * stride + 2 * NQ + qi * D +
                                                                c0 + 4 * half);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = cb + IL * u;
                if (c < cnt) {
                    const float w = wgt[c * NQ + qi];
                    acc.x += w * v[u].x;
                    acc.y += w * v[u].y;
                    acc.z += w * v[u].z;
                    acc.w += w * v[u].w;
                }
            }
        }
    }
    red4[il][f] = acc;
    __syncthreads();
    if (threadIdx.x < FPI && qi < G) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < IL; ++k) {
            const float4 x = red4[k][f];
            o.x += x.x; o.y += x.y; o.z += x.z; o.w += x.w;
        }
        const float inv = 1.f / lstar[qi];
        uint2 hv;
        hv.x = pack_h2(o.x * inv, o.y * inv);
        hv.y = pack_h2(o.z * inv, o.w * inv);
        *reinterpret_cast<uint2*>(p.out + ((int64_t)b * L.Hq + (int64_t)h * G + qi) * D + c0 + 4 * half) = hv;
    }
}

template <int D, int NQ>
int launch_decode_t(const Layout& L, const AttnParams& p, cudaStream_t s, const LaunchMarks& mk) {
    using C = Cfg<D, NQ>;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(decode_split_kernel<D, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        attr = true;
    }
    const int n_body = p.total_items - p.n_region_items;
    // the streaming decode kernel takes the body items (when it has an instance for the layout)
    // and, where it covers the layout, the region items too, in one launch; otherwise the region
    // items go through the generic kernel
    const bool streaming = body_ctas_per_sm(L) > 0;
    const bool fused_regions = streaming && region_kernel_ok(L);
    auto mark = [&](void* ev) -> bool {
        if (!ev) return true;
        if (mk.side) {
            if (cudaEventRecord((cudaEvent_t)mk.fork, s) != cudaSuccess) return false;
            if (cudaStreamWaitEvent((cudaStream_t)mk.side, (cudaEvent_t)mk.fork, 0) != cudaSuccess) return false;
            return cudaEventRecordWithFlags((cudaEvent_t)ev, (cudaStream_t)mk.side, mk.flags) == cudaSuccess;
        }
        return cudaEventRecordWithFlags((cudaEvent_t)ev, s, mk.flags) == cudaSuccess;
    };
    if (!mark(mk.before)) return (int)cudaErrorInvalidResourceHandle;
    if (streaming) {
        const int e = launch_decode_fused(L, p, n_body, fused_regions ? p.n_region_items : 0, s, mk.pdl);
        if (e != 0) return e;
    }
    if (p.n_region_items > 0 && !fused_regions) {
        // the remainder tiles (the area's last K_BYTES + V_BYTES) only for layouts that use them
        auto split_fmt = [](int f) { return qblock_bits(f) != 0 || f == KVQ_TURBO3 || f == KVQ_TQ5_0; };
        const bool lo = split_fmt(L.fmt[0]) || split_fmt(L.fmt[1]);
        const int smem = C::SMEM - (lo ? 0 : C::K_BYTES + C::V_BYTES);
        decode_split_kernel<D, NQ><<<p.n_region_items, kThreads, smem, s>>>(L, p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return (int)e;
    }
    if (!mark(mk.after)) return (int)cudaErrorInvalidResourceHandle;
    int max_cnt = 0;
    for (int i = 0; i < p.n_seq; ++i)
        max_cnt = max(max_cnt, p.seq[i].items_per_head + p.seq[i].body_per_head);
    if (max_cnt > kMergeMaxItems) return (int)cudaErrorInvalidConfiguration;
    dim3 mg(p.n_seq * L.H, D / 8);
    const size_t msmem = (size_t)max_cnt * NQ * 2 * sizeof(float);
    if (msmem > 48 * 1024)
        cudaFuncSetAttribute(decode_merge_kernel<D, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msmem);
    // programmatic serialization only where the launch ahead is the decode kernel (no event
    // record or generic kernel between them)
    const bool pdl = mk.pdl && streaming && fused_regions && (!mk.after || mk.side);
    const cudaError_t e = launch_k(decode_merge_kernel<D, NQ>, mg, dim3(256), msmem, s, pdl, L, p);
    return e != cudaSuccess ? (int)e : (int)cudaGetLastError();
}

}  // namespace

int upload_tables_attn(const FormatTables& t) {
    return (int)cudaMemcpyToSymbol(c_tab, &t, sizeof(FormatTables));
}

int launch_decode(const Layout& L, const AttnParams& p, void* stream, const LaunchMarks& mk) {
    if (p.total_items == 0) return 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (L.NQ == 8) {
        if (L.D == 128) return launch_decode_t<128, 8>(L, p, s, mk);
        if (L.D == 256) return launch_decode_t<256, 8>(L, p, s, mk);
        if (L.D == 512) return launch_decode_t<512, 8>(L, p, s, mk);
    } else {
        if (L.D == 128) return launch_decode_t<128, 16>(L, p, s, mk);
        if (L.D == 256) return launch_decode_t<256, 16>(L, p, s, mk);
        if (L.D == 512) return launch_decode_t<512, 16>(L, p, s, mk);
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace kvq

// ---------------------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// Some callers of this library have no way to call cudaMalloc: a host program that links
// only this C ABI inside a runtime whose memory manager has already reserved the device
// (an inference server's fixed pool), or a latency-critical loop where cudaMalloc's implicit
// synchronisation is not acceptable. kv_decode_attn needs a caller-provided workspace for
// its per-work-item partial results; kv_decode_attn_noalloc uses the fixed array below
// instead, so the caller passes only inputs and outputs.
//
// The array is a file-scope device variable: every GPU that loads this library holds its
// 32 MiB until the process exits. All calls share it and it keeps the last call's contents;
// nothing in it has to start at zero (each call writes every partial it later reads), and
// calls that overlap on the GPU (concurrent streams, or host threads racing) corrupt each
// other's partials. Its device address is looked up once per device, on the first call made
// with that device current; make that first call before any stream capture begins.
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;
}  // namespace
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

extern "C" kvq_status kv_decode_attn_noalloc(kvq_cache* cache, int layer, const int32_t* seq_ids, int n_seq,
                                             const void* q, void* out, void* stream) {
    using namespace kvq;
    const kvq_config* cfg = cache_config(cache);
    if (!cfg) return KVQ_EINVAL;
    size_t need = 0;
    kvq_status st = kv_required_bytes(cfg, nullptr, &need);
    if (st != KVQ_OK) return st;
    if (need > kNoAllocScratchBytes) return KVQ_EUNSUPPORTED;   // workspace would exceed the fixed 32 MiB
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ECUDA;
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!addr[dev]) {
            void* a = nullptr;
            if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || !a) return KVQ_ECUDA;
            addr[dev] = a;
        }
        ptr = addr[dev];
    }
    return kv_decode_attn(cache, layer, seq_ids, n_seq, q, out, ptr, kNoAllocScratchBytes, stream);
}
