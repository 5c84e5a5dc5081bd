// Codec kernels of the rotated low-bit KV cache: append (rotate + tq6_0 staging, exact
// copies) and dequant. The seals (TBQ4 / Q8_0 / Q4_0 and KVarN) are in kernels_seal.cu.
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

// ---------------------------------------------------------------------------- tq6_0
__device__ __forceinline__ int tq6_code_at(const uint8_t* blk, int j) {
    const int lo = (blk[j >> 1] >> ((j & 1) * 4)) & 15;
    const int hi = (blk[64 + (j >> 2)] >> ((j & 3) * 2)) & 3;
    return lo | (hi << 4);
}

// ---------------------------------------------------------------------------- append
// grid (n_seq * n_tok, H, 2), block D / 4 threads (one warp per 128 values); dynamic smem D bytes.
// Sequence b appends count[b] (<= n_tok) positions, read from its input rows src_off[b] on (the
// input holds src_stride rows per sequence).
__global__ void append_kernel(Layout L, AppendParams p) {
    extern __shared__ uint8_t cs[];                   // D codes
    const int b = blockIdx.x / p.n_tok, t = blockIdx.x % p.n_tok;
    if (t >= p.count[b]) return;
    const int h = blockIdx.y, w = blockIdx.z, D = L.D;
    const int pos = p.n0[b] + t;
    const uint16_t* src = (w ? p.v : p.k) + (((int64_t)b * p.src_stride + p.src_off[b] + t) * L.H + h) * D;
    // positions of one append that share a tail slot (pos mod T) would race: only the newest T
    // positions (pos >= tail_from) write it
    append_row(L, p.pool, L.unit(p.layer, p.slot[b], h), w, pos, src, pos >= p.tail_from[b],
               (int)threadIdx.x, (int)blockDim.x, cs);
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
            if (kvarn_bits(fmt)) {
                const int bits = kvarn_bits(fmt);
                const int hh = ch >> 8, j = ch & 255;
                const uint8_t* tr = rec + (int64_t)hh * (4096 * bits + 1152);
                const int code = (w == 0) ? kvarn_code(tr, bits, 256, t, j) : kvarn_code(tr, bits, 128, j, t);
                const uint16_t* sb = (const uint16_t*)(tr + 4096 * bits);
                x = fmul(fadd(fmul((float)code, h2f(sb[t])), h2f(sb[128 + t])), h2f(sb[256 + j]));
            } else if (fmt == KVQ_TURBO3) {   // token-major for K and V
                const int code = ((rec[t * (D / 4) + (ch >> 2)] >> (2 * (ch & 3))) & 3) |
                                 (((rec[32 * D + t * (D / 8) + (ch >> 3)] >> (ch & 7)) & 1) << 2);
                x = fmul(c_tab.cent3[code], h2f(((const uint16_t*)(rec + 48 * D))[t * (D / 128) + (ch >> 7)]));
            } else if (fmt == KVQ_TQ5_0) {     // token-major for K and V
                const int code = ((rec[t * (D / 2) + (ch >> 1)] >> ((ch & 1) * 4)) & 15) |
                                 (((rec[64 * D + t * (D / 8) + (ch >> 3)] >> (ch & 7)) & 1) << 4);
                x = fmul((float)(code - 16), h2f(((const uint16_t*)(rec + 80 * D))[t * (D / 128) + (ch >> 7)]));
            } else if (qblock_bits(fmt)) {   // token-major for K and V
                const int bits = qblock_bits(fmt);
                int code = (rec[t * (D / 2) + (ch >> 1)] >> ((ch & 1) * 4)) & 15;
                if (bits == 5) code |= ((rec[64 * D + t * (D / 8) + (ch >> 3)] >> (ch & 7)) & 1) << 4;
                else if (bits == 6) code |= ((rec[64 * D + t * (D / 4) + (ch >> 2)] >> (2 * (ch & 3))) & 3) << 4;
                const uint16_t* sc = (const uint16_t*)(rec + record_code_bytes(fmt, D));
                const float d = h2f(sc[t * (D / 32) + (ch >> 5)]);
                const int Lv = qblock_sym_levels(fmt);
                x = Lv ? fmul((float)(code - (Lv + 1)), d)
                       : fadd(fmul((float)code, d), h2f(sc[4 * D + t * (D / 32) + (ch >> 5)]));
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
