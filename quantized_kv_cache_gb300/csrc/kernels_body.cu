// Decode attention over sealed body records: the bandwidth-critical part of the path.
//
// One CTA per work item (sequence, KV head, run of 128-position groups). Warp 8 is a
// producer: it streams each group's K record and V record (contiguous, 16-byte multiples)
// into a ring of shared-memory stages with cp.async.bulk, completion tracked by mbarriers.
// Warps 0-7 consume each group in three phases separated by consumer-only barriers:
//   1. scores: warp w takes positions [16w, 16w+16) and all D channels, decoding its K rows
//      from shared memory straight into mma.sync m16n8k16 fragments (positions on M, the GQA
//      query group on N) against query fragments prepared once per group (KVarN: the column
//      scales folded in, q' = q C) or once per item;
//   2. softmax: warp per query over the group's 128 positions (log2 domain, running max and
//      sum); it writes P' = p x (value scale of the position) in fp16, laid out in mma
//      fragment order, one copy per value-scale block;
//   3. values: warp w takes channels [wD/8, (w+1)D/8) for all 128 positions, decoding V rows
//      (channel-major records: one 16-byte read covers 32 positions of a channel) into
//      fragments, O^T[ch][q] += V^T P'^T.
// Q8_0 / Q4_0 codes keep the fp16 exponent-trick offset (1024 + code is exact in fp16), removed
// once per group with the sum of the matching operand (sum q' for scores, sum P' for values);
// KVarN codes enter centred (code - 2^(b-1)), their zero point absorbing the centre. Scales: KVarN K row scale / zero point and TBQ4 / Q8_0 / Q4_0 K block
// scales in the score epilogue; V row / block scales in P'; KVarN V column scale and zero
// point once per group (O += C acc + C sum_t p_t (Z_t + 2^(b-1) S_t)).
// The partial (m, l, o) is rotated back to the original domain and merged with the region
// partials by decode_merge_kernel (kernels_attn.cu).
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

enum { KF_KVARN = 0, KF_TBQ4 = 1, KF_Q8 = 2, KF_Q4 = 3 };

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
// Bounded wait on an mbarrier phase. On timeout it sets bit 1 of the status word and the
// CTA's abort flag; once the flag is set no thread waits again (the CTA runs to its end on
// stale data, reaching every barrier, and the host learns of it from the status word).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status, volatile int* abort_flag) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtime();
    while (!mbar_try(bar, parity)) {
        if (*abort_flag) return false;
        if (gtime() - t0 > kWaitNs) {
            atomicOr(status, 2u);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
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

// ------------------------------------------------------------------------------ half2 decode
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t as_u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ uint32_t pack_f2(float a, float b) { return as_u(__floats2half2_rn(a, b)); }
// Nibbles x and x+4 of w (x = sh / 4) as half2 (1024 + code_x, 1024 + code_x+4), exact.
__device__ __forceinline__ uint32_t nibraw(uint32_t w, int sh) { return ((w >> sh) & 0x000F000Fu) | 0x64006400u; }
// Bits x and x+4 of w as half2 (0 or 1), exact.
__device__ __forceinline__ __half2 bit2(uint32_t w, int x) {
    const uint32_t t = w >> x;
    return __hsub2(as_h2((t & 1u) | ((t << 12) & 0x10000u) | 0x64006400u), as_h2(0x64006400u));
}
// Signed bytes of w (sel 0x5140: bytes 0,1; 0x7362: bytes 2,3) as half2 (1152 + b), exact.
__device__ __forceinline__ uint32_t i8raw(uint32_t w, uint32_t sel) {
    return __byte_perm(w ^ 0x80808080u, 0x64646464u, sel);
}

// ------------------------------------------------------------------------------ geometry
template <int D, int NQ, int KF, int VF, int KB, int VB>
struct Geo {
    static constexpr int NT = NQ / 8;
    static constexpr int KS = D / 16;                                   // score k-steps
    static constexpr int WK = (KF == KF_KVARN) ? 256 : (KF == KF_TBQ4 ? 128 : 32);   // K scale block
    static constexpr int NBK = D / WK;
    static constexpr int KSPB = WK / 16;                                // k-steps per K block
    static constexpr int WV = (VF == KF_KVARN) ? 256 : (VF == KF_TBQ4 ? 128 : 32);   // V scale block
    static constexpr int NVB = D / WV;                                  // P' copies
    static constexpr int MT = D / 128;                                  // value m-tiles per warp
    static constexpr bool KNIB = (KF == KF_KVARN || KF == KF_Q4);       // K pairs (x, x+4)
    static constexpr bool VNIB = (VF == KF_KVARN || VF == KF_Q4);
    static constexpr float KOFF = (KF == KF_Q8) ? 1152.f : (KF == KF_Q4 ? 1032.f : 0.f);
    static constexpr float VOFF = (VF == KF_Q8) ? 1152.f : (VF == KF_Q4 ? 1032.f : 0.f);
    // KVarN codes enter the mma centred (code - 2^(b-1), small exact integers): the row's zero
    // point then absorbs the centre, Z + 2^(b-1) S, and no large offset cancels in the sums
    static constexpr float KCEN = (KF == KF_KVARN) ? (float)(1 << (KB - 1)) : 0.f;
    static constexpr float VCEN = (VF == KF_KVARN) ? (float)(1 << (VB - 1)) : 0.f;
    static constexpr bool LUT = (KF == KF_TBQ4) || (VF == KF_TBQ4);
    // shared memory beyond the stages (bytes)
    static constexpr bool QHALF = NQ * D > 4096;                        // rotated query kept in fp16
    static constexpr int QR_BYTES = NQ * D * (QHALF ? 2 : 4);
    static constexpr int QB_BYTES = NT * KS * 32 * 8;                   // query fragments
    static constexpr int S_BYTES = 128 * NQ * 4;                        // scores of one group
    static constexpr int P_BYTES = NVB * NQ * 128 * 2;                  // P' copies
    static constexpr int ST_FLOATS = NQ * (4 + 2 * NVB + 2 * NBK);     // m, l, alpha, pad, psum, zsum, sumq, zq
    static constexpr int FIXED = 128 + (LUT ? kLutBytes : 0) + QR_BYTES + QB_BYTES + S_BYTES + P_BYTES + ST_FLOATS * 4;
};

// Index of position t inside one query's [kk][tq][4] P' row: the value k-step kk and slot e
// that thread quad tq feeds to the mma for that position (the V decoder's pairing).
template <bool VNIB>
__device__ __forceinline__ int pidx(int t) {
    const int tq = t >> 5, r = t & 31;
    int kk, e;
    if (VNIB) {    // nibble words of 8 positions, pairs (x, x+4), (x+1, x+5)
        const int m = r >> 3, rr = r & 7;
        kk = 2 * m + ((rr >> 1) & 1);
        e = ((rr & 1) << 1) | (rr >> 2);
    } else {       // natural pairs (2i, 2i+1)
        kk = r >> 2;
        e = r & 3;
    }
    return (kk * 4 + tq) * 4 + e;
}

// Channel of column e (0..3) of score k-step j for thread quad tq.
template <int KSPB, int WK, bool KNIB>
__device__ __forceinline__ int kchan(int j, int tq, int e) {
    const int b = j / KSPB, jj = j % KSPB;
    int c;
    if (KNIB) {
        const int cx = 8 * (jj >> 1) + 2 * (jj & 1);
        c = cx + ((e & 1) ? 4 : 0) + (e >> 1);
    } else {
        c = 4 * jj + e;
    }
    return b * WK + (WK / 4) * tq + c;
}

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

// ------------------------------------------------------------------------------ the kernel
template <int D, int NQ, int KF, int VF, int KB, int VB>
__global__ void __launch_bounds__(kBodyThreads, 1) decode_body_kernel(Layout L, AttnParams p, int nst) {
    using Gm = Geo<D, NQ, KF, VF, KB, VB>;
    constexpr int NT = Gm::NT, KS = Gm::KS, NBK = Gm::NBK, KSPB = Gm::KSPB, WK = Gm::WK;
    constexpr int NVB = Gm::NVB, WV = Gm::WV, MT = Gm::MT;
    extern __shared__ __align__(128) uint8_t smem[];

    // ---- work item: body items follow the region items
    const int item = p.n_region_items + (int)blockIdx.x;
    int b = 0;
    while (b + 1 < p.n_seq && p.seq[b + 1].body_first <= item) ++b;
    const SeqSpan& sp = p.seq[b];
    const int local = item - sp.body_first;
    const int h = local / sp.body_per_head;
    const int g0 = (local % sp.body_per_head) * p.body_chunk;
    const int ngroups = min(g0 + p.body_chunk, sp.body_groups) - g0;
    const int64_t unit = L.unit(p.layer, sp.slot, h);
    uint32_t* status = status_word(L, p.pool);

    const uint32_t recK = (uint32_t)L.rec_bytes[0], recV = (uint32_t)L.rec_bytes[1];
    const uint32_t v_off = (recK + 127u) & ~127u;
    const uint32_t stage_bytes = (v_off + recV + 127u) & ~127u;
    uint8_t* stages = smem;
    uint8_t* tailp = smem + (size_t)nst * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(tailp);
    uint64_t* empty = full + nst;
    uint8_t* cur = tailp + 128;
    uint32_t* lut = reinterpret_cast<uint32_t*>(cur);
    cur += Gm::LUT ? kLutBytes : 0;
    float* qr = reinterpret_cast<float*>(cur);            // fp32 rows, or fp16 rows when Gm::QHALF
    __half* qrh = reinterpret_cast<__half*>(cur);         cur += Gm::QR_BYTES;
    uint32_t* qb = reinterpret_cast<uint32_t*>(cur);      cur += Gm::QB_BYTES;
    float* sbuf = reinterpret_cast<float*>(cur);          cur += Gm::S_BYTES;
    __half* pbuf = reinterpret_cast<__half*>(cur);        cur += Gm::P_BYTES;
    float* stt = reinterpret_cast<float*>(cur);
    float* m_run = stt;                // [NQ]
    float* l_run = stt + NQ;           // [NQ]
    float* alpha = stt + 2 * NQ;       // [NQ]
    float* psum = stt + 4 * NQ;        // [NVB][NQ] offset x sum of P'
    float* zsum = psum + NVB * NQ;     // [NVB][NQ] sum of p Z (KVarN V)
    float* sumq = zsum + NVB * NQ;     // [NBK][NQ] offset x sum of the query fragments
    float* zq = sumq + NBK * NQ;       // [NBK][NQ] sum of the query fragments (KVarN zero point)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < nst; ++i) {
            mbar_init(su32(&full[i]), 1);
            mbar_init(su32(&empty[i]), kConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    // ================================================================== producer warp
    if (warp == kConsumers) {
        if (lane == 0) {
            const uint8_t* kb = body_rec(L, p.pool, 0, unit, g0);
            const uint8_t* vb = body_rec(L, p.pool, 1, unit, g0);
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < ngroups; ++i) {
                const int sl = i % nst;
                if (i >= nst) ok = mbar_wait(su32(&empty[sl]), ((i / nst) - 1) & 1, status, &s_abort);
                if (!ok) break;
                const uint32_t dst = su32(stages + (size_t)sl * stage_bytes);
                const uint32_t fb = su32(&full[sl]);
                mbar_expect_tx(fb, recK + recV);
                bulk_g2s(dst, kb + (size_t)i * recK, recK, fb);
                bulk_g2s(dst + v_off, vb + (size_t)i * recV, recV, fb);
                ++issued;
            }
            if (!ok) {   // a wait timed out: wait (bounded, fresh limit) for copies still in flight
                s_abort = 0;
                for (int i = max(0, issued - nst); i < issued; ++i)
                    mbar_wait(su32(&full[i % nst]), (i / nst) & 1, status, &s_abort);
            }
        }
        return;
    }

    // ================================================================== consumers: set-up
    const int g = lane >> 2, tq = lane & 3;
    const int G = L.G;
    if (Gm::LUT) {
        for (int i = threadIdx.x; i < 256 * 32; i += kCT) {
            const int by = i >> 5;
            lut[i] = pack_f2(c_tab.cent[by & 15], c_tab.cent[by >> 4]);
        }
    }
    {   // rotated query rows (one warp per rotation block of a row)
        const uint16_t* q = p.q + ((int64_t)b * L.Hq + (int64_t)h * G) * D;
        const int rot = L.rot;
        if (rot == ROT_HAD256) {
            if constexpr (D >= 256) {
                for (int u = warp; u < NQ * (D / 256); u += kConsumers) {
                    const int rr = u / (D / 256), c0 = (u % (D / 256)) * 256;
                    float v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[k] = (rr < G) ? h2f(q[rr * D + c0 + lane + 32 * k]) : 0.f;
                    warp_rotate<8>(v, lane, rot);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if constexpr (Gm::QHALF) qrh[rr * D + c0 + lane + 32 * k] = __float2half_rn(v[k]);
                        else qr[rr * D + c0 + lane + 32 * k] = v[k];
                    }
                }
            }
        } else {
            for (int u = warp; u < NQ * (D / 128); u += kConsumers) {
                const int rr = u / (D / 128), c0 = (u % (D / 128)) * 128;
                float v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] = (rr < G) ? h2f(q[rr * D + c0 + lane + 32 * k]) : 0.f;
                warp_rotate<4>(v, lane, rot);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if constexpr (Gm::QHALF) qrh[rr * D + c0 + lane + 32 * k] = __float2half_rn(v[k]);
                    else qr[rr * D + c0 + lane + 32 * k] = v[k];
                }
            }
        }
        if (threadIdx.x < NQ) {
            m_run[threadIdx.x] = -INFINITY;
            l_run[threadIdx.x] = 0.f;
        }
    }
    csync();

    // query fragments: entry (nt, j, g, tq) holds, for query nt*8+g, the 4 channels of the
    // column slots of thread (g, tq) in score k-step j (KVarN: times the group's column scale)
    auto build_qb = [&](const uint8_t* krec) {
        for (int e = threadIdx.x; e < NT * KS * 32; e += kCT) {
            const int tq_ = e & 3, g_ = (e >> 2) & 7, j = (e >> 5) % KS, nt = (e >> 5) / KS;
            const int qi = nt * 8 + g_;
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = kchan<KSPB, WK, Gm::KNIB>(j, tq_, k);
                float x;
                if constexpr (Gm::QHALF) x = __half2float(qrh[qi * D + c]);
                else x = qr[qi * D + c];
                if (KF == KF_KVARN) {
                    const uint16_t* sb =
                        reinterpret_cast<const uint16_t*>(krec + (c >> 8) * (4096 * KB + 1152) + 4096 * KB);
                    x *= h2f(sb[256 + (c & 255)]);
                }
                v[k] = x;
            }
            uint2 u;
            u.x = pack_f2(v[0], v[1]);
            u.y = pack_f2(v[2], v[3]);
            reinterpret_cast<uint2*>(qb)[e] = u;
        }
        csync();
        // per query and K block: the sum of the rounded fragments, times the decode offset
        // (and plain, for the KVarN zero point); one warp per (block, query)
        for (int u = warp; u < NBK * NQ; u += kConsumers) {
            const int bk = u / NQ, qi = u % NQ;
            const int nt = qi / 8, g_ = qi % 8;
            float s = 0.f;
            for (int e = lane; e < KSPB * 4; e += 32) {
                const int j = bk * KSPB + e / 4, tq_ = e & 3;
                const uint2 uu = reinterpret_cast<const uint2*>(qb)[((nt * KS + j) * 8 + g_) * 4 + tq_];
                const float2 a = __half22float2(as_h2(uu.x)), c2 = __half22float2(as_h2(uu.y));
                s += (a.x + a.y) + (c2.x + c2.y);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) {
                sumq[bk * NQ + qi] = s * Gm::KOFF;
                zq[bk * NQ + qi] = s;
            }
        }
        csync();
    };
    if (KF != KF_KVARN) build_qb(nullptr);

    float O[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) O[mt][nt][i] = 0.f;
    const float sc = L.scale * kLog2e;
    const uint2* qb2 = reinterpret_cast<const uint2*>(qb);
    const uint2* pb2 = reinterpret_cast<const uint2*>(pbuf);

    for (int gi = 0; gi < ngroups; ++gi) {
        const int sl = gi % nst;
        mbar_wait(su32(&full[sl]), (gi / nst) & 1, status, &s_abort);
        const uint8_t* kr = stages + (size_t)sl * stage_bytes;
        const uint8_t* vr = kr + v_off;
        if (KF == KF_KVARN) build_qb(kr);

        // ---------------- phase 1: scores of positions [16 warp, 16 warp + 16), all channels
        {
            const int t0 = 16 * warp + g, t1 = t0 + 8;
            float acc[NBK][NT][4];
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[bk][nt][0] = acc[bk][nt][1] = acc[bk][nt][2] = acc[bk][nt][3] = 0.f;
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk) {
                if (KF == KF_KVARN) {
                    // this thread's 64 channels of the 256-channel tile bk: 32 bytes per row; odd
                    // rows read the two halves in the other order so a quarter warp hits 32 banks
                    const uint8_t* tb = kr + (size_t)bk * (4096 * KB + 1152);
                    const int odd = g & 1;
                    uint4 x0a = *reinterpret_cast<const uint4*>(tb + t0 * 128 + 32 * tq + 16 * odd);
                    uint4 x0b = *reinterpret_cast<const uint4*>(tb + t0 * 128 + 32 * tq + 16 * (1 - odd));
                    uint4 x1a = *reinterpret_cast<const uint4*>(tb + t1 * 128 + 32 * tq + 16 * odd);
                    uint4 x1b = *reinterpret_cast<const uint4*>(tb + t1 * 128 + 32 * tq + 16 * (1 - odd));
                    if (odd) {
                        const uint4 t = x0a; x0a = x0b; x0b = t;
                        const uint4 u = x1a; x1a = x1b; x1b = u;
                    }
                    const uint32_t W0[8] = {x0a.x, x0a.y, x0a.z, x0a.w, x0b.x, x0b.y, x0b.z, x0b.w};
                    const uint32_t W1[8] = {x1a.x, x1a.y, x1a.z, x1a.w, x1b.x, x1b.y, x1b.z, x1b.w};
                    uint2 H0 = make_uint2(0, 0), H1 = make_uint2(0, 0);
                    if (KB == 5) {
                        H0 = *reinterpret_cast<const uint2*>(tb + 16384 + t0 * 32 + 8 * tq);
                        H1 = *reinterpret_cast<const uint2*>(tb + 16384 + t1 * 32 + 8 * tq);
                    }
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int m = jj >> 1, sh = 8 * (jj & 1);
                        uint32_t a0 = nibraw(W0[m], sh), a2 = nibraw(W0[m], sh + 4);
                        uint32_t a1 = nibraw(W1[m], sh), a3 = nibraw(W1[m], sh + 4);
                        if (KB == 5) {
                            const int x = 8 * m + 2 * (jj & 1);
                            const uint32_t h0 = (x < 32) ? H0.x : H0.y, h1 = (x < 32) ? H1.x : H1.y;
                            const __half2 s16 = __float2half2_rn(16.f);
                            a0 = as_u(__hfma2(bit2(h0, x & 31), s16, as_h2(a0)));
                            a2 = as_u(__hfma2(bit2(h0, (x & 31) + 1), s16, as_h2(a2)));
                            a1 = as_u(__hfma2(bit2(h1, x & 31), s16, as_h2(a1)));
                            a3 = as_u(__hfma2(bit2(h1, (x & 31) + 1), s16, as_h2(a3)));
                        }
                        {   // 1024 + code  ->  code - 2^(b-1)
                            const __half2 off = __float2half2_rn(1024.f + Gm::KCEN);
                            a0 = as_u(__hsub2(as_h2(a0), off)); a1 = as_u(__hsub2(as_h2(a1), off));
                            a2 = as_u(__hsub2(as_h2(a2), off)); a3 = as_u(__hsub2(as_h2(a3), off));
                        }
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt], a0, a1, a2, a3, bq.x, bq.y);
                        }
                    }
                } else if (KF == KF_TBQ4) {
                    // blocks of 128 channels: 16 bytes of this row and block per thread
                    const uint4 y0 = *reinterpret_cast<const uint4*>(kr + t0 * (D / 2) + 64 * bk + 16 * tq);
                    const uint4 y1 = *reinterpret_cast<const uint4*>(kr + t1 * (D / 2) + 64 * bk + 16 * tq);
                    const uint32_t W0[4] = {y0.x, y0.y, y0.z, y0.w}, W1[4] = {y1.x, y1.y, y1.z, y1.w};
                    const uint32_t* lt = lut + lane;
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int m = jj >> 1, sh = 16 * (jj & 1);
                        const uint32_t a0 = lt[((W0[m] >> sh) & 0xFF) * 32], a2 = lt[((W0[m] >> (sh + 8)) & 0xFF) * 32];
                        const uint32_t a1 = lt[((W1[m] >> sh) & 0xFF) * 32], a3 = lt[((W1[m] >> (sh + 8)) & 0xFF) * 32];
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt], a0, a1, a2, a3, bq.x, bq.y);
                        }
                    }
                } else if (KF == KF_Q8) {
                    const uint2 x0 = *reinterpret_cast<const uint2*>(kr + t0 * D + 32 * bk + 8 * tq);
                    const uint2 x1 = *reinterpret_cast<const uint2*>(kr + t1 * D + 32 * bk + 8 * tq);
                    const uint32_t W0[2] = {x0.x, x0.y}, W1[2] = {x1.x, x1.y};
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const uint32_t a0 = i8raw(W0[jj], 0x5140), a2 = i8raw(W0[jj], 0x7362);
                        const uint32_t a1 = i8raw(W1[jj], 0x5140), a3 = i8raw(W1[jj], 0x7362);
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt], a0, a1, a2, a3, bq.x, bq.y);
                        }
                    }
                } else {   // Q4_0 K
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(kr + t0 * (D / 2) + 16 * bk + 4 * tq);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(kr + t1 * (D / 2) + 16 * bk + 4 * tq);
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int sh = 8 * (jj & 1);
                        const uint32_t a0 = nibraw(w0, sh), a2 = nibraw(w0, sh + 4);
                        const uint32_t a1 = nibraw(w1, sh), a3 = nibraw(w1, sh + 4);
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt], a0, a1, a2, a3, bq.x, bq.y);
                        }
                    }
                }
            }
            // epilogue: s = sum over K blocks of e(t) (acc - off sum q') + z(t) sum q'
            float s4[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) s4[nt][0] = s4[nt][1] = s4[nt][2] = s4[nt][3] = 0.f;
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk) {
                float e0, e1, z0 = 0.f, z1 = 0.f;
                if (KF == KF_KVARN) {
                    const uint16_t* sb =
                        reinterpret_cast<const uint16_t*>(kr + (size_t)bk * (4096 * KB + 1152) + 4096 * KB);
                    e0 = h2f(sb[t0]); e1 = h2f(sb[t1]);
                    z0 = h2f(sb[128 + t0]) + Gm::KCEN * e0;
                    z1 = h2f(sb[128 + t1]) + Gm::KCEN * e1;
                } else if (KF == KF_TBQ4) {
                    const uint16_t* nr = reinterpret_cast<const uint16_t*>(kr + 64 * D);
                    e0 = h2f(nr[t0 * (D / 128) + bk]); e1 = h2f(nr[t1 * (D / 128) + bk]);
                } else {
                    const uint16_t* dr = reinterpret_cast<const uint16_t*>(kr + (KF == KF_Q8 ? 128 : 64) * D);
                    e0 = h2f(dr[t0 * (D / 32) + bk]); e1 = h2f(dr[t1 * (D / 32) + bk]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int qc = nt * 8 + 2 * tq;
                    const float o0 = sumq[bk * NQ + qc], o1 = sumq[bk * NQ + qc + 1];
                    const float y0 = zq[bk * NQ + qc], y1 = zq[bk * NQ + qc + 1];
                    s4[nt][0] += e0 * (acc[bk][nt][0] - o0) + z0 * y0;
                    s4[nt][1] += e0 * (acc[bk][nt][1] - o1) + z0 * y1;
                    s4[nt][2] += e1 * (acc[bk][nt][2] - o0) + z1 * y0;
                    s4[nt][3] += e1 * (acc[bk][nt][3] - o1) + z1 * y1;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int qc = nt * 8 + 2 * tq;
                sbuf[t0 * NQ + qc] = s4[nt][0] * sc;
                sbuf[t0 * NQ + qc + 1] = s4[nt][1] * sc;
                sbuf[t1 * NQ + qc] = s4[nt][2] * sc;
                sbuf[t1 * NQ + qc + 1] = s4[nt][3] * sc;
            }
        }
        csync();

        // ---------------- phase 2: softmax over the group, P' copies in fragment order
        for (int qi = warp; qi < NQ; qi += kConsumers) {
            float sv[4];
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                sv[i] = sbuf[(lane + 32 * i) * NQ + qi];
                mx = fmaxf(mx, sv[i]);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mo = m_run[qi];
            const float mn = fmaxf(mo, mx);
            const float a = exp2f(mo - mn);
            float ls = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                sv[i] = exp2f(sv[i] - mn);
                ls += sv[i];
            }
            float ps[NVB], zs[NVB];
#pragma unroll
            for (int v = 0; v < NVB; ++v) {
                ps[v] = 0.f;
                zs[v] = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = lane + 32 * i;
                    float f;
                    if (VF == KF_KVARN) {
                        const uint16_t* sb =
                            reinterpret_cast<const uint16_t*>(vr + (size_t)v * (4096 * VB + 1152) + 4096 * VB);
                        f = h2f(sb[t]);
                        zs[v] += sv[i] * (h2f(sb[128 + t]) + Gm::VCEN * f);
                    } else if (VF == KF_TBQ4) {
                        f = h2f(reinterpret_cast<const uint16_t*>(vr + 64 * D)[t * (D / 128) + v]);
                    } else {
                        f = h2f(reinterpret_cast<const uint16_t*>(vr + (VF == KF_Q8 ? 128 : 64) * D)[t * (D / 32) + v]);
                    }
                    const __half ph = __float2half_rn(sv[i] * f);
                    pbuf[((size_t)v * NQ + qi) * 128 + pidx<Gm::VNIB>(t)] = ph;
                    ps[v] += __half2float(ph);
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                ls += __shfl_xor_sync(0xffffffffu, ls, o);
#pragma unroll
                for (int v = 0; v < NVB; ++v) {
                    ps[v] += __shfl_xor_sync(0xffffffffu, ps[v], o);
                    zs[v] += __shfl_xor_sync(0xffffffffu, zs[v], o);
                }
            }
            if (lane == 0) {
                m_run[qi] = mn;
                l_run[qi] = l_run[qi] * a + ls;
                alpha[qi] = a;
#pragma unroll
                for (int v = 0; v < NVB; ++v) {
                    psum[v * NQ + qi] = ps[v] * Gm::VOFF;
                    zsum[v * NQ + qi] = zs[v];
                }
            }
        }
        csync();

        // ---------------- phase 3: O^T[ch][q] += V^T P'^T for channels [w D/8, (w+1) D/8)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int c0 = warp * (D / 8) + 16 * mt + g, c1 = c0 + 8;
            const int v = (warp * (D / 8) + 16 * mt) / WV;
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            uint32_t X0[8], X1[8];
            uint32_t H0 = 0, H1 = 0;
            const uint8_t* vt = vr;
            if (VF == KF_KVARN) {
                vt = vr + (size_t)(c0 >> 8) * (4096 * VB + 1152);
                const uint4 y0 = *reinterpret_cast<const uint4*>(vt + (c0 & 255) * 64 + 16 * tq);
                const uint4 y1 = *reinterpret_cast<const uint4*>(vt + (c1 & 255) * 64 + 16 * tq);
                X0[0] = y0.x; X0[1] = y0.y; X0[2] = y0.z; X0[3] = y0.w;
                X1[0] = y1.x; X1[1] = y1.y; X1[2] = y1.z; X1[3] = y1.w;
                if (VB == 5) {
                    H0 = *reinterpret_cast<const uint32_t*>(vt + 16384 + (c0 & 255) * 16 + 4 * tq);
                    H1 = *reinterpret_cast<const uint32_t*>(vt + 16384 + (c1 & 255) * 16 + 4 * tq);
                }
            } else if (VF == KF_TBQ4 || VF == KF_Q4) {
                const uint4 y0 = *reinterpret_cast<const uint4*>(vr + c0 * 64 + 16 * tq);
                const uint4 y1 = *reinterpret_cast<const uint4*>(vr + c1 * 64 + 16 * tq);
                X0[0] = y0.x; X0[1] = y0.y; X0[2] = y0.z; X0[3] = y0.w;
                X1[0] = y1.x; X1[1] = y1.y; X1[2] = y1.z; X1[3] = y1.w;
            } else {   // Q8_0: 32 positions = 32 bytes of the channel row; odd rows swap halves (banks)
                const int odd = g & 1;
                uint4 y0a = *reinterpret_cast<const uint4*>(vr + c0 * 128 + 32 * tq + 16 * odd);
                uint4 y0b = *reinterpret_cast<const uint4*>(vr + c0 * 128 + 32 * tq + 16 * (1 - odd));
                uint4 y1a = *reinterpret_cast<const uint4*>(vr + c1 * 128 + 32 * tq + 16 * odd);
                uint4 y1b = *reinterpret_cast<const uint4*>(vr + c1 * 128 + 32 * tq + 16 * (1 - odd));
                if (odd) {
                    const uint4 t = y0a; y0a = y0b; y0b = t;
                    const uint4 u = y1a; y1a = y1b; y1b = u;
                }
                X0[0] = y0a.x; X0[1] = y0a.y; X0[2] = y0a.z; X0[3] = y0a.w;
                X0[4] = y0b.x; X0[5] = y0b.y; X0[6] = y0b.z; X0[7] = y0b.w;
                X1[0] = y1a.x; X1[1] = y1a.y; X1[2] = y1a.z; X1[3] = y1a.w;
                X1[4] = y1b.x; X1[5] = y1b.y; X1[6] = y1b.z; X1[7] = y1b.w;
            }
            const uint32_t* lt = lut + lane;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t a0, a1, a2, a3;
                if (Gm::VNIB) {
                    const int m = kk >> 1, sh = 8 * (kk & 1);
                    a0 = nibraw(X0[m], sh); a2 = nibraw(X0[m], sh + 4);
                    a1 = nibraw(X1[m], sh); a3 = nibraw(X1[m], sh + 4);
                    if (VF == KF_KVARN && VB == 5) {
                        const int x = 8 * m + 2 * (kk & 1);
                        const __half2 s16 = __float2half2_rn(16.f);
                        a0 = as_u(__hfma2(bit2(H0, x), s16, as_h2(a0)));
                        a2 = as_u(__hfma2(bit2(H0, x + 1), s16, as_h2(a2)));
                        a1 = as_u(__hfma2(bit2(H1, x), s16, as_h2(a1)));
                        a3 = as_u(__hfma2(bit2(H1, x + 1), s16, as_h2(a3)));
                    }
                    if (VF == KF_KVARN) {   // 1024 + code  ->  code - 2^(b-1)
                        const __half2 off = __float2half2_rn(1024.f + Gm::VCEN);
                        a0 = as_u(__hsub2(as_h2(a0), off)); a1 = as_u(__hsub2(as_h2(a1), off));
                        a2 = as_u(__hsub2(as_h2(a2), off)); a3 = as_u(__hsub2(as_h2(a3), off));
                    }
                } else if (VF == KF_TBQ4) {
                    const int m = kk >> 1, sh = 16 * (kk & 1);
                    a0 = lt[((X0[m] >> sh) & 0xFF) * 32]; a2 = lt[((X0[m] >> (sh + 8)) & 0xFF) * 32];
                    a1 = lt[((X1[m] >> sh) & 0xFF) * 32]; a3 = lt[((X1[m] >> (sh + 8)) & 0xFF) * 32];
                } else {
                    a0 = i8raw(X0[kk], 0x5140); a2 = i8raw(X0[kk], 0x7362);
                    a1 = i8raw(X1[kk], 0x5140); a3 = i8raw(X1[kk], 0x7362);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint2 bp = pb2[(((size_t)v * NQ + nt * 8 + g) * 8 + kk) * 4 + tq];
                    mma16816(acc[nt], a0, a1, a2, a3, bp.x, bp.y);
                }
            }
            // O = alpha O + F (acc - off sum P' + sum p Z)
            float F0 = 1.f, F1 = 1.f;
            if (VF == KF_KVARN) {
                const uint16_t* sb = reinterpret_cast<const uint16_t*>(vt + 4096 * VB);
                F0 = h2f(sb[256 + (c0 & 255)]);
                F1 = h2f(sb[256 + (c1 & 255)]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int qc = nt * 8 + 2 * tq;
                const float al0 = alpha[qc], al1 = alpha[qc + 1];
                const float ps0 = psum[v * NQ + qc], ps1 = psum[v * NQ + qc + 1];
                float z0 = 0.f, z1 = 0.f;
                if (VF == KF_KVARN) {
                    z0 = zsum[v * NQ + qc];
                    z1 = zsum[v * NQ + qc + 1];
                }
                O[mt][nt][0] = al0 * O[mt][nt][0] + F0 * (acc[nt][0] - ps0 + z0);
                O[mt][nt][1] = al1 * O[mt][nt][1] + F0 * (acc[nt][1] - ps1 + z1);
                O[mt][nt][2] = al0 * O[mt][nt][2] + F1 * (acc[nt][2] - ps0 + z0);
                O[mt][nt][3] = al1 * O[mt][nt][3] + F1 * (acc[nt][3] - ps1 + z1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&empty[sl]));
    }

    // ---- partial: o rotated back to the original domain, m and l
    csync();
    float* ofin = reinterpret_cast<float*>(stages);                     // [NQ][D], stages drained
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int c0 = warp * (D / 8) + 16 * mt + g;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int qc = nt * 8 + 2 * tq;
            ofin[qc * D + c0] = O[mt][nt][0];
            ofin[(qc + 1) * D + c0] = O[mt][nt][1];
            ofin[qc * D + c0 + 8] = O[mt][nt][2];
            ofin[(qc + 1) * D + c0 + 8] = O[mt][nt][3];
        }
    }
    csync();
    inverse_rotate_c(ofin, NQ, D, L.rot);
    float* part = p.partials + (size_t)item * (2 * NQ + NQ * D);
    if (threadIdx.x < NQ) {
        part[threadIdx.x] = m_run[threadIdx.x];
        part[NQ + threadIdx.x] = l_run[threadIdx.x];
    }
    float4* po = reinterpret_cast<float4*>(part + 2 * NQ);
    const float4* o4 = reinterpret_cast<const float4*>(ofin);
    for (int e = threadIdx.x; e < NQ * D / 4; e += kCT) po[e] = o4[e];
}

// ------------------------------------------------------------------------------ launch
template <int D, int NQ, int KF, int VF, int KB, int VB>
int nstages(const Layout& L) {
    using Gm = Geo<D, NQ, KF, VF, KB, VB>;
    const uint32_t recK = (uint32_t)L.rec_bytes[0], recV = (uint32_t)L.rec_bytes[1];
    const size_t stage = ((((recK + 127u) & ~127u) + recV + 127u) & ~127u);
    const size_t budget = 227 * 1024;
    if ((size_t)Gm::FIXED >= budget) return 0;
    int nst = (int)((budget - Gm::FIXED) / stage);
    if (nst > 4) nst = 4;
    if ((size_t)nst * stage < (size_t)NQ * D * 4) return 0;      // the final rows reuse the stages
    return nst >= 2 ? nst : 0;
}

template <int D, int NQ, int KF, int VF, int KB, int VB>
int launch_t(const Layout& L, const AttnParams& p, int n_body, cudaStream_t st) {
    using Gm = Geo<D, NQ, KF, VF, KB, VB>;
    const int nst = nstages<D, NQ, KF, VF, KB, VB>(L);
    if (nst == 0) return (int)cudaErrorInvalidConfiguration;
    const uint32_t recK = (uint32_t)L.rec_bytes[0], recV = (uint32_t)L.rec_bytes[1];
    const size_t stage = ((((recK + 127u) & ~127u) + recV + 127u) & ~127u);
    const size_t smem = (size_t)nst * stage + Gm::FIXED;
    cudaFuncSetAttribute(decode_body_kernel<D, NQ, KF, VF, KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    decode_body_kernel<D, NQ, KF, VF, KB, VB><<<n_body, kBodyThreads, smem, st>>>(L, p, nst);
    return (int)cudaGetLastError();
}

// Instantiated combinations (head_dim, query tile, K format, V format); other layouts keep
// their body positions in the region kernel's generic path.
template <typename F>
int dispatch(const Layout& L, F&& f) {
    const int k = L.fmt[0], v = L.fmt[1];
#define KVQ_BODY_CASE(D_, NQ_, KF_, VF_, KB_, VB_, KFMT, VFMT) \
    if (L.D == D_ && L.NQ == NQ_ && k == KFMT && v == VFMT) return f.template run<D_, NQ_, KF_, VF_, KB_, VB_>();
    KVQ_BODY_CASE(128, 8, KF_TBQ4, KF_TBQ4, 4, 4, KVQ_TBQ4, KVQ_TBQ4)
    KVQ_BODY_CASE(256, 8, KF_TBQ4, KF_TBQ4, 4, 4, KVQ_TBQ4, KVQ_TBQ4)
    KVQ_BODY_CASE(256, 16, KF_TBQ4, KF_TBQ4, 4, 4, KVQ_TBQ4, KVQ_TBQ4)
    KVQ_BODY_CASE(128, 8, KF_Q8, KF_Q4, 4, 4, KVQ_Q8_0, KVQ_Q4_0)
    KVQ_BODY_CASE(128, 16, KF_Q8, KF_Q4, 4, 4, KVQ_Q8_0, KVQ_Q4_0)
    KVQ_BODY_CASE(256, 8, KF_KVARN, KF_KVARN, 4, 4, KVQ_KVARN4, KVQ_KVARN4)
    KVQ_BODY_CASE(256, 16, KF_KVARN, KF_KVARN, 4, 4, KVQ_KVARN4, KVQ_KVARN4)
    KVQ_BODY_CASE(512, 8, KF_KVARN, KF_KVARN, 5, 5, KVQ_KVARN5, KVQ_KVARN5)
    KVQ_BODY_CASE(512, 16, KF_KVARN, KF_KVARN, 5, 5, KVQ_KVARN5, KVQ_KVARN5)
#undef KVQ_BODY_CASE
    return -1;
}

struct NstFn {
    const Layout& L;
    template <int D, int NQ, int KF, int VF, int KB, int VB>
    int run() { return nstages<D, NQ, KF, VF, KB, VB>(L); }
};
struct LaunchFn {
    const Layout& L;
    const AttnParams& p;
    int n;
    cudaStream_t s;
    template <int D, int NQ, int KF, int VF, int KB, int VB>
    int run() { return launch_t<D, NQ, KF, VF, KB, VB>(L, p, n, s); }
};

}  // namespace

int upload_tables_body(const FormatTables& t) {
    return (int)cudaMemcpyToSymbol(c_tab, &t, sizeof(FormatTables));
}

// 1 when the body kernel has an instance for this layout (and its stages fit), else 0.
int body_ctas_per_sm(const Layout& L) {
    NstFn f{L};
    const int r = dispatch(L, f);
    return r > 0 ? 1 : 0;
}

// Launches the body kernel over the body items (those after the region items of p).
int launch_decode_body(const Layout& L, const AttnParams& p, int n_body, void* stream) {
    if (n_body <= 0) return 0;
    LaunchFn f{L, p, n_body, (cudaStream_t)stream};
    const int r = dispatch(L, f);
    return r < 0 ? (int)cudaErrorInvalidValue : r;
}

}  // namespace kvq
