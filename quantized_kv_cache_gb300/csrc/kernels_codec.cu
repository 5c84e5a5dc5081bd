// Codec kernels of the rotated low-bit KV cache: append (rotate + tq6_0 staging, exact
// copies), the KVarN seal and dequant. The TBQ4 / Q8_0 / Q4_0 seal is in kernels_seal.cu.
//
// Every floating-point step uses the explicit round-to-nearest intrinsics (__fadd_rn,
// __fmul_rn, __fdiv_rn, __fsqrt_rn) and this file is built with -fmad=false, so no
// multiply-add is contracted and records are reproducible bit for bit: one IEEE fp32
// rounding per operation, halving-tree sums, round-half-even rint and fp16/bf16 casts.
#include <cuda_runtime.h>
#include "append_row.cuh"

namespace kvq {
namespace {

using namespace codec;

__device__ __forceinline__ float warp_min(float v) {
    for (int s = 16; s >= 1; s >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, s));
    return v;
}
// Last five levels of a halving-tree sum whose 32 partials sit one per lane: level
// stride 16 adds lane i + 16 onto lane i, and so on; every lane ends with the total.
__device__ __forceinline__ float warp_tree_tail(float v) {
    for (int s = 16; s >= 1; s >>= 1) v = fadd(v, __shfl_xor_sync(kFull, v, s));
    return v;
}

// ---------------------------------------------------------------------------- FWHT
// Butterflies of a Sylvester-order FWHT over blocks of n values in shared memory,
// strides ascending; executed by the whole thread block.
__device__ void block_fwht(float* xs, int total, int n) {
    for (int s = 1; s < n; s <<= 1) {
        for (int p = threadIdx.x; p < total / 2; p += blockDim.x) {
            const int blk = p / (n / 2), q = p % (n / 2);
            const int i = blk * n + (q / s) * 2 * s + (q % s);
            const float a = xs[i], b = xs[i + s];
            xs[i] = fadd(a, b);
            xs[i + s] = fsub(a, b);
        }
        __syncthreads();
    }
}

__device__ void block_rotate(float* xs, int D, int rot) {
    if (rot == ROT_HAD256) {
        block_fwht(xs, D, 256);
        for (int i = threadIdx.x; i < D; i += blockDim.x) xs[i] = fmul(xs[i], kHad256Scale);
        __syncthreads();
    } else if (rot == ROT_TBQ128) {
        for (int i = threadIdx.x; i < D; i += blockDim.x)
            if (sign_neg(0, i & 127)) xs[i] = -xs[i];
        __syncthreads();
        block_fwht(xs, D, 128);
        for (int i = threadIdx.x; i < D; i += blockDim.x) {
            float y = xs[i];
            if (sign_neg(1, i & 127)) y = -y;
            xs[i] = fmul(y, kTbqScale);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------- tq6_0
__device__ __forceinline__ int tq6_code_at(const uint8_t* blk, int j) {
    const int lo = (blk[j >> 1] >> ((j & 1) * 4)) & 15;
    const int hi = (blk[64 + (j >> 2)] >> ((j & 3) * 2)) & 3;
    return lo | (hi << 4);
}

// Values of channels c0 + lane + 32 k (k < NK) of journal position pos in the body's
// domain: tq6_0 rows are dequantized (already rotated at append), exact rows are widened
// and rotated here (NK covers whole rotation blocks: 4 for TBQ128, 8 for HAD256).
template <int NK>
__device__ __forceinline__ void load_journal_row(const Layout& L, const void* pool, int w, int64_t unit,
                                                 int pos, int c0, int lane, float (&v)[NK]) {
    const int slot = journal_slot(L, pos);
    if (L.journal == KVQ_TQ6_0) {
        const uint8_t* row = jcode_row(L, pool, w, unit, slot);
        const uint16_t* sc = jscale_row(L, pool, w, unit, slot);
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const int c = c0 + lane + 32 * k;
            const int b = c >> 7, j = c & 127;
            const float d = h2f(sc[b]);
            v[k] = fmul((float)(tq6_code_at(row + 96 * b, j) - 32), d);
        }
        return;
    }
    const uint16_t* row = jexact_row(L, pool, w, unit, slot);
#pragma unroll
    for (int k = 0; k < NK; ++k) v[k] = x16_to_f(row[c0 + lane + 32 * k], L.journal);
    if (L.rot == ROT_HAD256) {
        if constexpr (NK % 8 == 0) {
            // one or more 256-blocks: k in [8m, 8m+8) is block m
#pragma unroll
            for (int m = 0; m < NK / 8; ++m) {
                float t[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) t[k] = v[8 * m + k];
                warp_fwht<8>(t, lane);
#pragma unroll
                for (int k = 0; k < 8; ++k) v[8 * m + k] = fmul(t[k], kHad256Scale);
            }
        }
    } else if (L.rot == ROT_TBQ128) {
        if constexpr (NK % 4 == 0) {
#pragma unroll
            for (int m = 0; m < NK / 4; ++m) {
                float t[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = lane + 32 * k;
                    t[k] = sign_neg(0, j) ? -v[4 * m + k] : v[4 * m + k];
                }
                warp_fwht<4>(t, lane);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = lane + 32 * k;
                    const float y = sign_neg(1, j) ? -t[k] : t[k];
                    v[4 * m + k] = fmul(y, kTbqScale);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------- append
// grid (n_seq * n_tok, H, 2), block D / 4 threads (one warp per 128 values); dynamic smem D bytes.
__global__ void append_kernel(Layout L, AppendParams p) {
    extern __shared__ uint8_t cs[];                   // D codes
    const int b = blockIdx.x / p.n_tok, t = blockIdx.x % p.n_tok;
    const int h = blockIdx.y, w = blockIdx.z, D = L.D;
    const int pos = p.n0[b] + t;
    const uint16_t* src = (w ? p.v : p.k) + (((int64_t)b * p.n_tok + t) * L.H + h) * D;
    // positions of one append that share a tail slot (pos mod T) would race: only the newest T
    // positions of the append write it
    append_row(L, p.pool, L.unit(p.layer, p.slot[b], h), w, pos, src, pos + L.T >= p.n0[b] + p.n_tok,
               (int)threadIdx.x, (int)blockDim.x, cs);
}

// ---------------------------------------------------------------------------- KVarN seal
// One 128 x 256 tile (SJ-KVaRN §2.2): HAD256-rotated journal rows, 16 alternating
// row/column passes of spread balancing, per-row b-bit rounding with fp16 scales.
// grid (groups, H, 2 * D/256), 512 threads; dynamic smem: Y [128][257] fp32 (padded so
// row and column walks are bank-conflict free) + codes [128][256] bytes.
constexpr int kYS = 257;

__device__ __forceinline__ void kvarn_row(const Layout& L, const void* pool, int w, int64_t unit,
                                          int pos, int half, int lane, float (&v)[8]) {
    load_journal_row<8>(L, pool, w, unit, pos, 256 * half, lane, v);
}

__global__ void __launch_bounds__(512) seal_kvarn_kernel(Layout L, SealParams p) {
    const SealTaskPos tk = seal_task(p, blockIdx.x);
    const int nh = L.D / 256;
    const int h = blockIdx.y, w = blockIdx.z / nh, half = blockIdx.z % nh;
    const int fmt = L.fmt[w];
    const int bits = (fmt == KVQ_KVARN5) ? 5 : 4;
    const float Q = (float)((1 << bits) - 1);
    const int64_t unit = L.unit(tk.layer, tk.slot, h);
    extern __shared__ float Y[];                           // [128][kYS]
    uint8_t* codes = (uint8_t*)(Y + 128 * kYS);            // [128][256]
    __shared__ float r[128], c[256], invS[128], Zs[128], invC[256];
    __shared__ uint16_t S16[128], Z16[128], C16[256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int NW = 16;

    for (int t = warp; t < 128; t += NW) {
        float v[8];
        kvarn_row(L, p.pool, w, unit, tk.pos0 + t, half, lane, v);
#pragma unroll
        for (int k = 0; k < 8; ++k) Y[t * kYS + lane + 32 * k] = v[k];
        if (lane == 0) r[t] = 1.f;
    }
    for (int j = threadIdx.x; j < 256; j += blockDim.x) c[j] = 1.f;
    __syncthreads();

    for (int pass = 0; pass < 16; ++pass) {
        if ((pass & 1) == 0) {
            for (int t = warp; t < 128; t += NW) {
                float v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = Y[t * kYS + lane + 32 * k];
                // halving tree over 256: strides 128, 64, 32 in-lane, then 16..1
                float a0 = fadd(v[0], v[4]), a1 = fadd(v[1], v[5]), a2 = fadd(v[2], v[6]), a3 = fadd(v[3], v[7]);
                a0 = fadd(a0, a2); a1 = fadd(a1, a3);
                const float mu = fmul(warp_tree_tail(fadd(a0, a1)), 1.0f / 256.0f);
                float e[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) { const float d = fsub(v[k], mu); e[k] = fmul(d, d); }
                a0 = fadd(e[0], e[4]); a1 = fadd(e[1], e[5]); a2 = fadd(e[2], e[6]); a3 = fadd(e[3], e[7]);
                a0 = fadd(a0, a2); a1 = fadd(a1, a3);
                const float var = fmul(warp_tree_tail(fadd(a0, a1)), 1.0f / 256.0f);
                float sig = __fsqrt_rn(var);
                if (sig <= 9.5367431640625e-07f) sig = 1.f;     // 2^-20
                const float inv = fdiv(1.0f, sig);
#pragma unroll
                for (int k = 0; k < 8; ++k) Y[t * kYS + lane + 32 * k] = fmul(v[k], inv);
                if (lane == 0) r[t] = fmul(r[t], sig);
            }
        } else {
            for (int j = warp; j < 256; j += NW) {
                float v[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) v[m] = Y[(lane + 32 * m) * kYS + j];
                // halving tree over 128 rows: strides 64, 32 in-lane, then 16..1
                const float mu = fmul(warp_tree_tail(fadd(fadd(v[0], v[2]), fadd(v[1], v[3]))), 1.0f / 128.0f);
                float e[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) { const float d = fsub(v[m], mu); e[m] = fmul(d, d); }
                const float var = fmul(warp_tree_tail(fadd(fadd(e[0], e[2]), fadd(e[1], e[3]))), 1.0f / 128.0f);
                float sig = __fsqrt_rn(var);
                if (sig <= 9.5367431640625e-07f) sig = 1.f;
                const float inv = fdiv(1.0f, sig);
#pragma unroll
                for (int m = 0; m < 4; ++m) Y[(lane + 32 * m) * kYS + j] = fmul(v[m], inv);
                if (lane == 0) c[j] = fmul(c[j], sig);
            }
        }
        __syncthreads();
    }

    // row rounding parameters
    for (int t = warp; t < 128; t += NW) {
        float lo = 3.4e38f, hi = -3.4e38f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float y = Y[t * kYS + lane + 32 * k];
            lo = fminf(lo, y);
            hi = fmaxf(hi, y);
        }
        lo = warp_min(lo);
        hi = warp_max(hi);
        if (lane == 0) {
            const uint16_t s16 = f2h_bits(fdiv(fmul(r[t], fsub(hi, lo)), Q));
            const uint16_t z16 = f2h_bits(fmul(r[t], lo));
            S16[t] = s16;
            Z16[t] = z16;
            const float s = h2f(s16);
            invS[t] = (s == 0.f) ? 0.f : fdiv(1.0f, s);
            Zs[t] = h2f(z16);
            flag_nonfinite(L, p.pool, s);
            flag_nonfinite(L, p.pool, Zs[t]);
        }
    }
    for (int j = threadIdx.x; j < 256; j += blockDim.x) {
        const uint16_t c16 = f2h_bits(c[j]);
        C16[j] = c16;
        invC[j] = fdiv(1.0f, h2f(c16));
        flag_nonfinite(L, p.pool, h2f(c16));
    }
    __syncthreads();

    // codes from the input tile (re-read; identical bits) and the stored scales
    for (int t = warp; t < 128; t += NW) {
        float v[8];
        kvarn_row(L, p.pool, w, unit, tk.pos0 + t, half, lane, v);
        const float is = invS[t], z = Zs[t];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int j = lane + 32 * k;
            float q = 0.f;
            if (is != 0.f) {
                q = rintf(fmul(fsub(fmul(v[k], invC[j]), z), is));
                q = fminf(fmaxf(q, 0.f), Q);
            }
            codes[t * 256 + j] = (uint8_t)q;
        }
    }
    __syncthreads();

    uint8_t* rec = body_rec(L, p.pool, w, unit, tk.g) + (int64_t)half * (4096 * bits + 1152);
    if (w == 0) {           // K: token-major low plane [128][128], high plane [128][32]
        for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
            const int t = i >> 7, j = 2 * (i & 127);
            rec[i] = (uint8_t)((codes[t * 256 + j] & 15) | ((codes[t * 256 + j + 1] & 15) << 4));
        }
        if (bits == 5) {
            for (int i = threadIdx.x; i < 128 * 32; i += blockDim.x) {
                const int t = i >> 5, j0 = 8 * (i & 31);
                uint8_t b = 0;
#pragma unroll
                for (int m = 0; m < 8; ++m) b |= (uint8_t)(((codes[t * 256 + j0 + m] >> 4) & 1) << m);
                rec[16384 + i] = b;
            }
        }
    } else {                // V: channel-major low plane [256][64], high plane [256][16]
        for (int i = threadIdx.x; i < 256 * 64; i += blockDim.x) {
            const int j = i >> 6, t = 2 * (i & 63);
            rec[i] = (uint8_t)((codes[t * 256 + j] & 15) | ((codes[(t + 1) * 256 + j] & 15) << 4));
        }
        if (bits == 5) {
            for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
                const int j = i >> 4, t0 = 8 * (i & 15);
                uint8_t b = 0;
#pragma unroll
                for (int m = 0; m < 8; ++m) b |= (uint8_t)(((codes[(t0 + m) * 256 + j] >> 4) & 1) << m);
                rec[16384 + i] = b;
            }
        }
    }
    uint16_t* sb = (uint16_t*)(rec + 4096 * bits);
    for (int i = threadIdx.x; i < 576; i += blockDim.x) {
        uint16_t x = 0;
        if (i < 128) x = S16[i];
        else if (i < 256) x = Z16[i - 128];
        else if (i < 512) x = C16[i - 256];
        sb[i] = x;
    }
}

// ---------------------------------------------------------------------------- dequant
// kind: RegionKind of the positions [p0, p0 + n); out fp32 [n][D].
__global__ void dequant_kernel(Layout L, const void* pool, int layer, int slot, int head, int w, int kind,
                               int64_t p0, int64_t n, float* out) {
    const int64_t total = n * L.D;
    const int64_t unit = L.unit(layer, slot, head);
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int pos = (int)(p0 + e / L.D);
        const int ch = (int)(e % L.D);
        float x = 0.f;
        if (kind == RK_SINK) {
            x = h2f(sink_row(L, pool, w, unit, pos)[ch]);
        } else if (kind == RK_TAIL) {
            x = x16_to_f(tail_row(L, pool, w, unit, pos % L.T)[ch], L.tail_fmt);
        } else if (kind == RK_JEXACT) {
            x = x16_to_f(jexact_row(L, pool, w, unit, journal_slot(L, pos))[ch], L.journal);
        } else if (kind == RK_RING) {
            const int s = journal_slot(L, pos);
            const int b = ch >> 7;
            x = fmul((float)(tq6_code_at(jcode_row(L, pool, w, unit, s) + 96 * b, ch & 127) - 32),
                     h2f(jscale_row(L, pool, w, unit, s)[b]));
        } else {  // body
            const int g = (pos - kSink) / kGroup, t = (pos - kSink) % kGroup;
            const uint8_t* rec = body_rec(L, pool, w, unit, g);
            const int fmt = L.fmt[w];
            const int D = L.D;
            if (fmt == KVQ_KVARN4 || fmt == KVQ_KVARN5) {
                const int bits = (fmt == KVQ_KVARN5) ? 5 : 4;
                const int hh = ch >> 8, j = ch & 255;
                const uint8_t* tr = rec + (int64_t)hh * (4096 * bits + 1152);
                int code;
                if (w == 0) {
                    code = (tr[t * 128 + (j >> 1)] >> ((j & 1) * 4)) & 15;
                    if (bits == 5) code |= ((tr[16384 + t * 32 + (j >> 3)] >> (j & 7)) & 1) << 4;
                } else {
                    code = (tr[j * 64 + (t >> 1)] >> ((t & 1) * 4)) & 15;
                    if (bits == 5) code |= ((tr[16384 + j * 16 + (t >> 3)] >> (t & 7)) & 1) << 4;
                }
                const uint16_t* sb = (const uint16_t*)(tr + 4096 * bits);
                x = fmul(fadd(fmul((float)code, h2f(sb[t])), h2f(sb[128 + t])), h2f(sb[256 + j]));
            } else {
                const int64_t cb = record_code_bytes(fmt, D);
                const uint16_t* sc = (const uint16_t*)(rec + cb);
                if (fmt == KVQ_Q8_0) {
                    const int8_t q = (int8_t)(w == 0 ? rec[t * D + ch] : rec[ch * 128 + t]);
                    x = fmul((float)q, h2f(sc[t * (D / 32) + (ch >> 5)]));
                } else {
                    int code;
                    if (w == 0) code = (rec[t * (D / 2) + (ch >> 1)] >> ((ch & 1) * 4)) & 15;
                    else code = (rec[ch * 64 + (t >> 1)] >> ((t & 1) * 4)) & 15;
                    if (fmt == KVQ_Q4_0) x = fmul((float)(code - 8), h2f(sc[t * (D / 32) + (ch >> 5)]));
                    else x = fmul(c_tab.cent[code], h2f(sc[t * (D / 128) + (ch >> 7)]));
                }
            }
        }
        out[e] = x;
    }
}

}  // namespace

int upload_tables_codec(const FormatTables& t) {
    return (int)cudaMemcpyToSymbol(c_tab, &t, sizeof(FormatTables));
}

int launch_append(const Layout& L, const AppendParams& p, void* stream) {
    dim3 grid(p.n_seq * p.n_tok, L.H, 2);
    const int threads = L.D / 4;
    const size_t smem = (size_t)L.D;
    append_kernel<<<grid, threads, smem, (cudaStream_t)stream>>>(L, p);
    return (int)cudaGetLastError();
}

int launch_seal(const Layout& L, const SealParams& p, void* stream) {
    const int groups = p.n_layers * p.groups_per_layer;
    if (groups == 0) return 0;
    cudaStream_t s = (cudaStream_t)stream;
    const bool kvarn = (L.fmt[0] == KVQ_KVARN4 || L.fmt[0] == KVQ_KVARN5);
    if (kvarn) {
        const size_t smem = 128 * kYS * sizeof(float) + 128 * 256;
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(seal_kvarn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            attr = true;
        }
        dim3 grid(groups, L.H, 2 * (L.D / 256));
        seal_kvarn_kernel<<<grid, 512, smem, s>>>(L, p);
        return (int)cudaGetLastError();
    }
    return launch_seal_rows(L, p, stream);   // TBQ4, Q8_0, Q4_0 (kernels_seal.cu)
}

int launch_dequant(const Layout& L, const void* pool, int layer, int slot, int head, int which, int kind,
                        int64_t p0, int64_t n, float* out, void* stream) {
    if (n <= 0) return 0;
    const int64_t total = n * L.D;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    dequant_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(L, pool, layer, slot, head, which, kind, p0, n, out);
    return (int)cudaGetLastError();
}

}  // namespace kvq
