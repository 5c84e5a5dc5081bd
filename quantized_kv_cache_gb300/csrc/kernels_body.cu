// Decode attention over sealed body records: the bandwidth-critical part of the path.
//
// One CTA per work item (sequence, KV head, run of 128-position groups). Warp 8 is a
// producer: it streams each group's K record and V record (contiguous, 16-byte multiples)
// into a ring of shared-memory stages with cp.async.bulk, completion tracked by mbarriers.
// Warps 0-7 are consumers: they decode the packed codes straight from shared memory into
// mma.sync m16n8k16 register fragments (no fp16 copy of the cache anywhere) and run
//   S^T[pos][q] = K Q^T      (positions on M, the GQA query group on N)
//   O^T[ch][q] += V^T P^T    (channels on M)
// with an online softmax in the log2 domain. Warps form teams of D/128 (each warp owns 128
// channels); a team shares 16-position tiles and adds its partial scores through shared
// memory. Scales are applied where they are cheapest and exact in algebra:
//   KVarN K: column scales C folded into the query (q' = q C), row scale and zero point in the
//            score epilogue (s = S_t (q'.code) + Z_t sum(q'));
//   KVarN V: column scale multiplied into the decoded codes, row scale into P (p S_t), the zero
//            point added once per group (O += C sum_t p_t Z_t);
//   TBQ4:    centroids looked up per byte from a lane-replicated table, norms into the score
//            epilogue (K) or P (V);
//   Q8_0/Q4_0: per-32 scales multiplied into the decoded K values or into P (V).
// The inverse rotation of the partial output, the partial format and the merge are those of
// the region kernel (kernels_attn.cu).
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cfloat>
#include "device_common.cuh"

namespace kvq {
namespace {

constexpr int kConsumers = 8;
constexpr int kBodyThreads = (kConsumers + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTbqScale = 0.0883883461356163f;
constexpr int kLutBytes = 256 * 32 * 4;
constexpr uint64_t kWaitNs = 2000000000ull;   // bounded waits: 2 s, then the status word is set

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
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(r) : "r"(x));
    return r;
}

// ------------------------------------------------------------------------------ half2 decode
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t as_u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ uint32_t pack_f2(float a, float b) { return as_u(__floats2half2_rn(a, b)); }

// Nibbles x and x+4 of w (x = sh/4) as the exact half2 (code_x, code_{x+4}).
__device__ __forceinline__ __half2 nib2(uint32_t w, int sh) {
    return __hsub2(as_h2(((w >> sh) & 0x000F000Fu) | 0x64006400u), as_h2(0x64006400u));
}
// Bits x and x+4 of w as half2 (0/1).
__device__ __forceinline__ __half2 bit2(uint32_t w, int x) {
    const uint32_t t = w >> x;
    return __hsub2(as_h2((t & 1u) | ((t << 12) & 0x10000u) | 0x64006400u), as_h2(0x64006400u));
}
// Signed bytes of w selected by sel (0x5140: bytes 0,1; 0x7362: bytes 2,3) as exact half2.
__device__ __forceinline__ __half2 i8pair(uint32_t w, uint32_t sel) {
    return __hsub2(as_h2(__byte_perm(w ^ 0x80808080u, 0x64646464u, sel)), as_h2(0x64806480u));
}

enum { KF_KVARN = 0, KF_TBQ4 = 1, KF_Q8 = 2, KF_Q4 = 3 };

__device__ __forceinline__ int fmt_kind(int fmt) {
    if (fmt == KVQ_TBQ4) return KF_TBQ4;
    if (fmt == KVQ_Q8_0) return KF_Q8;
    if (fmt == KVQ_Q4_0) return KF_Q4;
    return KF_KVARN;
}

// Token offset (within a thread's run of positions) of slot e of tile a, by the V decoder's
// pairing of positions inside one mma k-step (pairs must match the V^T fragment).
//  vp 0: nibble words of 8 positions, pairs (x, x+4)         (KVarN / Q4_0 V, >= 8 positions)
//  vp 1: natural pairs (2i, 2i+1)                             (TBQ4 / Q8_0 V)
//  vp 2: nibble pairs (0,2), (1,3) of a 4-position run       (KVarN / Q4_0 V, 4 positions)
__device__ __forceinline__ int tok_off(int vp, int a, int e) {
    if (vp == 1) return 4 * a + e;
    if (vp == 2) return (e & 1) * 2 + (e >> 1);
    return 8 * (a >> 1) + 2 * (a & 1) + (e & 1) * 4 + (e >> 1);
}

template <int D, int NQ>
struct BodyCfg {
    static constexpr int CS = D / 128;             // warps per team (channel slices)
    static constexpr int TEAMS = kConsumers / CS;
    static constexpr int TPT = CS;                 // 16-position tiles per team per group
    static constexpr int NT = NQ / 8;
    static constexpr int RUN = 4 * TPT;            // positions a thread owns per group
    static constexpr int SX_FLOATS = TEAMS * TPT * CS * 16 * NQ;       // partial scores exchange
    static constexpr bool QHALF = NQ * D > 4096;                        // keep the rotated query in fp16
    static constexpr int Q_BYTES = NQ * D * (QHALF ? 2 : 4);
};

// Shared state of one CTA.
struct BodySmem {
    uint8_t* stage;        // NST stages of [K record | V record]
    uint32_t stage_bytes;
    uint32_t v_off;
    int nst;
    uint64_t* full;
    uint64_t* empty;
    uint32_t* lut;         // [256][32] half2 pairs (TBQ4), or null
    void* qr;              // [NQ][D] rotated query, fp32 (or fp16 when large)
    float* sx;             // partial scores exchange
};

// Block-wide FWHT over rows (consumer warps only, synchronised by named barrier 9).
__device__ void fwht_rows_c(float* xs, int total, int n) {
    for (int s = 1; s < n; s <<= 1) {
        for (int p = threadIdx.x; p < total / 2; p += kConsumers * 32) {
            const int blk = p / (n / 2), q = p % (n / 2);
            const int i = blk * n + (q / s) * 2 * s + (q % s);
            const float a = xs[i], b = xs[i + s];
            xs[i] = a + b;
            xs[i + s] = a - b;
        }
        named_sync(9, kConsumers * 32);
    }
}

__device__ void rotate_rows_c(float* xs, int rows, int D, int rot, bool inverse) {
    const int total = rows * D;
    const int nthr = kConsumers * 32;
    if (rot == ROT_HAD256) {
        fwht_rows_c(xs, total, 256);
        for (int i = threadIdx.x; i < total; i += nthr) xs[i] *= 0.0625f;
        named_sync(9, nthr);
    } else if (rot == ROT_TBQ128) {
        const int first = inverse ? 1 : 0;
        for (int i = threadIdx.x; i < total; i += nthr)
            if (sign_neg(first, i & 127)) xs[i] = -xs[i];
        named_sync(9, nthr);
        fwht_rows_c(xs, total, 128);
        for (int i = threadIdx.x; i < total; i += nthr) {
            float y = xs[i];
            if (sign_neg(1 - first, i & 127)) y = -y;
            xs[i] = y * kTbqScale;
        }
        named_sync(9, nthr);
    }
}

// Forward rotation of one 2^k block (n = 32 NK values, value i = lane + 32 k in v[k]) of a
// query row, with warp shuffles: FWHT butterflies (strides ascending), then the scale (and,
// for TBQ128, the sign flips around it).
template <int NK>
__device__ __forceinline__ void warp_rotate(float (&v)[NK], int lane, int rot) {
    if (rot == ROT_NONE) return;
    if (rot == ROT_TBQ128) {
#pragma unroll
        for (int k = 0; k < NK; ++k)
            if (sign_neg(0, lane + 32 * k)) v[k] = -v[k];
    }
#pragma unroll
    for (int st = 1; st < 32; st <<= 1) {
        const bool upper = lane & st;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            const float o = __shfl_xor_sync(0xffffffffu, v[k], st);
            v[k] = upper ? (o - v[k]) : (v[k] + o);
        }
    }
#pragma unroll
    for (int m = 1; m < NK; m <<= 1)
#pragma unroll
        for (int k = 0; k < NK; ++k) {
            if (k & m) continue;
            const float a = v[k], b = v[k + m];
            v[k] = a + b;
            v[k + m] = a - b;
        }
#pragma unroll
    for (int k = 0; k < NK; ++k) {
        if (rot == ROT_HAD256) v[k] *= 0.0625f;
        else if (rot == ROT_TBQ128) v[k] = (sign_neg(1, lane + 32 * k) ? -v[k] : v[k]) * kTbqScale;
    }
}

// ------------------------------------------------------------------------------ the kernel
template <int D, int NQ>
__global__ void __launch_bounds__(kBodyThreads, 1) decode_body_kernel(Layout L, AttnParams p, int nst) {
    using C = BodyCfg<D, NQ>;
    constexpr int CS = C::CS, TPT = C::TPT, NT = C::NT, RUN = C::RUN;
    extern __shared__ __align__(128) uint8_t smem[];

    // ---- which work item: body items follow the region items
    const int item = p.n_region_items + (int)blockIdx.x;
    int b = 0;
    while (b + 1 < p.n_seq && p.seq[b + 1].body_first <= item) ++b;
    const SeqSpan& sp = p.seq[b];
    const int local = item - sp.body_first;
    const int h = local / sp.body_per_head;
    const int cidx = local % sp.body_per_head;
    const int g0 = cidx * p.body_chunk;
    const int g1 = min(g0 + p.body_chunk, sp.body_groups);
    const int ngroups = g1 - g0;
    const int64_t unit = L.unit(p.layer, sp.slot, h);
    uint32_t* status = status_word(L, p.pool);

    const int kk = fmt_kind(L.fmt[0]), vk = fmt_kind(L.fmt[1]);
    const int kbits = (L.fmt[0] == KVQ_KVARN5) ? 5 : 4, vbits = (L.fmt[1] == KVQ_KVARN5) ? 5 : 4;
    const uint32_t recK = (uint32_t)L.rec_bytes[0], recV = (uint32_t)L.rec_bytes[1];
    const uint32_t v_off = (recK + 127u) & ~127u;
    const uint32_t stage_bytes = (v_off + recV + 127u) & ~127u;
    const bool use_lut = (kk == KF_TBQ4) || (vk == KF_TBQ4);

    BodySmem S;
    S.stage = smem;
    S.stage_bytes = stage_bytes;
    S.nst = nst;
    uint8_t* tail_area = smem + (size_t)nst * stage_bytes;
    S.full = reinterpret_cast<uint64_t*>(tail_area);
    S.empty = S.full + nst;
    uint8_t* after_bars = tail_area + 128;
    S.lut = use_lut ? reinterpret_cast<uint32_t*>(after_bars) : nullptr;
    S.qr = after_bars + (use_lut ? kLutBytes : 0);
    S.sx = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(S.qr) + C::Q_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < nst; ++i) {
            mbar_init(su32(&S.full[i]), 1);
            mbar_init(su32(&S.empty[i]), kConsumers);
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
            for (int i = 0; i < ngroups && ok; ++i) {
                const int sl = i % nst;
                if (i >= nst) ok = mbar_wait(su32(&S.empty[sl]), ((i / nst) - 1) & 1, status, &s_abort);
                if (!ok) break;
                const uint32_t dst = su32(S.stage + (size_t)sl * stage_bytes);
                const uint32_t fb = su32(&S.full[sl]);
                mbar_expect_tx(fb, recK + recV);
                bulk_g2s(dst, kb + (size_t)i * recK, recK, fb);
                bulk_g2s(dst + v_off, vb + (size_t)i * recV, recV, fb);
                ++issued;
            }
            if (!ok) {
                // a wait timed out: wait (bounded, fresh limit) for the copies still in flight
                s_abort = 0;
                for (int i = max(0, issued - nst); i < issued; ++i)
                    mbar_wait(su32(&S.full[i % nst]), (i / nst) & 1, status, &s_abort);
            }
        }
        return;
    }

    // ================================================================== consumers
    const int T = warp / CS, s = warp % CS;
    const int g = lane >> 2, tq = lane & 3;
    const int G = L.G;
    const int vp = (vk == KF_TBQ4 || vk == KF_Q8) ? 1 : (RUN >= 8 ? 0 : 2);
    const int base = 16 * CS * T + RUN * tq;              // this thread's first position in a group

    if (use_lut) {
        for (int i = threadIdx.x; i < 256 * 32; i += kConsumers * 32) {
            const int by = i >> 5;
            S.lut[i] = pack_f2(c_tab.cent[by & 15], c_tab.cent[by >> 4]);
        }
    }
    const uint16_t* q = p.q + ((int64_t)b * L.Hq + (int64_t)h * G) * D;
    {
        constexpr int BLK = 128;                           // rotation work unit: 128 values
        const int rot = L.rot;
        const int unit_n = (rot == ROT_HAD256) ? 256 : BLK;
        const int units = NQ * (D / unit_n);
        for (int u = warp; u < units; u += kConsumers) {
            const int rr = u / (D / unit_n), c0 = (u % (D / unit_n)) * unit_n;
            if (unit_n == 256) {
                float v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = (rr < G) ? h2f(q[rr * D + c0 + lane + 32 * k]) : 0.f;
                warp_rotate<8>(v, lane, rot);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if constexpr (C::QHALF) reinterpret_cast<__half*>(S.qr)[rr * D + c0 + lane + 32 * k] = __float2half_rn(v[k]);
                    else reinterpret_cast<float*>(S.qr)[rr * D + c0 + lane + 32 * k] = v[k];
                }
            } else {
                float v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] = (rr < G) ? h2f(q[rr * D + c0 + lane + 32 * k]) : 0.f;
                warp_rotate<4>(v, lane, rot);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if constexpr (C::QHALF) reinterpret_cast<__half*>(S.qr)[rr * D + c0 + lane + 32 * k] = __float2half_rn(v[k]);
                    else reinterpret_cast<float*>(S.qr)[rr * D + c0 + lane + 32 * k] = v[k];
                }
            }
        }
    }
    named_sync(9, kConsumers * 32);

    // B fragments of the query for this thread's 32 channels (query g of every n-tile)
    const int cbase = 128 * s + 32 * tq;                  // first channel this thread contracts
    uint32_t qb[8][NT][2];
    float sumq[NT];                                        // sum of q' over the slice (KVarN), per query g
    auto build_qb = [&](const uint8_t* kscale) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int qoff = (nt * 8 + g) * D + cbase;
            auto qv = [&](int c) -> float {
                if constexpr (C::QHALF) return __half2float(reinterpret_cast<const __half*>(S.qr)[qoff + c]);
                else return reinterpret_cast<const float*>(S.qr)[qoff + c];
            };
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int c0, c1, c2, c3;
                if (kk == KF_KVARN || kk == KF_Q4) {
                    const int cx = 8 * (j >> 1) + 2 * (j & 1);
                    c0 = cx; c1 = cx + 4; c2 = cx + 1; c3 = cx + 5;
                } else {
                    c0 = 4 * j; c1 = 4 * j + 1; c2 = 4 * j + 2; c3 = 4 * j + 3;
                }
                float v0 = qv(c0), v1 = qv(c1), v2 = qv(c2), v3 = qv(c3);
                if (kscale) {
                    const uint16_t* Cc = reinterpret_cast<const uint16_t*>(kscale) + 256 + ((cbase & 255));
                    v0 *= h2f(Cc[c0]); v1 *= h2f(Cc[c1]); v2 *= h2f(Cc[c2]); v3 *= h2f(Cc[c3]);
                }
                qb[j][nt][0] = pack_f2(v0, v1);
                qb[j][nt][1] = pack_f2(v2, v3);
                if (kscale) {   // sum of q' as rounded for the mma, so the zero-point term matches
                    const float2 r0 = __half22float2(as_h2(qb[j][nt][0])), r1 = __half22float2(as_h2(qb[j][nt][1]));
                    acc += (r0.x + r0.y) + (r1.x + r1.y);
                }
            }
            if (kscale) {
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            }
            sumq[nt] = acc;
        }
    };
    if (kk != KF_KVARN) build_qb(nullptr);

    float m_run[NT][2], l_run[NT][2];
    float O[8][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) O[mt][nt][i] = 0.f;
    }
    const float sc = L.scale * kLog2e;
    const uint32_t ktile = 4096u * kbits + 1152u, vtile = 4096u * vbits + 1152u;

    for (int gi = 0; gi < ngroups; ++gi) {
        const int sl = gi % nst;
        mbar_wait(su32(&S.full[sl]), (gi / nst) & 1, status, &s_abort);
        const uint8_t* kr = S.stage + (size_t)sl * stage_bytes;
        const uint8_t* vr = kr + v_off;
        // per-slice views of the records
        const uint8_t* kt = kr + (kk == KF_KVARN ? (size_t)(s >> 1) * ktile : 0);   // KVarN 256-channel tile
        const uint8_t* vt = vr + (vk == KF_KVARN ? (size_t)(s >> 1) * vtile : 0);
        const uint8_t* ksb = kt + 4096u * kbits;                                     // KVarN scale block
        const uint8_t* vsb = vt + 4096u * vbits;
        if (kk == KF_KVARN) build_qb(ksb);

        // ---------------- scores of this team's tiles, partial over this warp's slice
        float* sxb = S.sx;
#pragma unroll
        for (int a = 0; a < TPT; ++a) {
            const int tk0 = base - RUN * tq + RUN * (g >> 1) + tok_off(vp, a, g & 1);
            const int tk1 = base - RUN * tq + RUN * (g >> 1) + tok_off(vp, a, 2 + (g & 1));
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            if (kk == KF_KVARN || kk == KF_Q4) {
                uint4 w0, w1;
                uint32_t h0 = 0, h1 = 0;
                float d0 = 1.f, d1 = 1.f;
                if (kk == KF_KVARN) {
                    w0 = *reinterpret_cast<const uint4*>(kt + tk0 * 128 + 64 * (s & 1) + 16 * tq);
                    w1 = *reinterpret_cast<const uint4*>(kt + tk1 * 128 + 64 * (s & 1) + 16 * tq);
                    if (kbits == 5) {
                        h0 = *reinterpret_cast<const uint32_t*>(kt + 16384 + tk0 * 32 + 16 * (s & 1) + 4 * tq);
                        h1 = *reinterpret_cast<const uint32_t*>(kt + 16384 + tk1 * 32 + 16 * (s & 1) + 4 * tq);
                    }
                } else {
                    w0 = *reinterpret_cast<const uint4*>(kr + tk0 * (D / 2) + 64 * s + 16 * tq);
                    w1 = *reinterpret_cast<const uint4*>(kr + tk1 * (D / 2) + 64 * s + 16 * tq);
                    const uint16_t* dr = reinterpret_cast<const uint16_t*>(kr + 64 * D);
                    d0 = h2f(dr[tk0 * (D / 32) + 4 * s + tq]);
                    d1 = h2f(dr[tk1 * (D / 32) + 4 * s + tq]);
                }
                const uint32_t W0[4] = {w0.x, w0.y, w0.z, w0.w}, W1[4] = {w1.x, w1.y, w1.z, w1.w};
                const __half2 d0h = __float2half2_rn(d0), d1h = __float2half2_rn(d1);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int m = j >> 1, sh = 8 * (j & 1);
                    __half2 a0 = nib2(W0[m], sh), a2 = nib2(W0[m], sh + 4);
                    __half2 a1 = nib2(W1[m], sh), a3 = nib2(W1[m], sh + 4);
                    if (kk == KF_KVARN && kbits == 5) {
                        const int x = 8 * m + 2 * (j & 1);
                        const __half2 sixteen = __float2half2_rn(16.f);
                        a0 = __hfma2(bit2(h0, x), sixteen, a0);
                        a2 = __hfma2(bit2(h0, x + 1), sixteen, a2);
                        a1 = __hfma2(bit2(h1, x), sixteen, a1);
                        a3 = __hfma2(bit2(h1, x + 1), sixteen, a3);
                    }
                    if (kk == KF_Q4) {
                        const __half2 eight = __float2half2_rn(8.f);
                        a0 = __hmul2(__hsub2(a0, eight), d0h);
                        a2 = __hmul2(__hsub2(a2, eight), d0h);
                        a1 = __hmul2(__hsub2(a1, eight), d1h);
                        a3 = __hmul2(__hsub2(a3, eight), d1h);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816(acc[nt], as_u(a0), as_u(a1), as_u(a2), as_u(a3), qb[j][nt][0], qb[j][nt][1]);
                }
            } else if (kk == KF_TBQ4) {
                const uint4 w0 = *reinterpret_cast<const uint4*>(kr + tk0 * (D / 2) + 64 * s + 16 * tq);
                const uint4 w1 = *reinterpret_cast<const uint4*>(kr + tk1 * (D / 2) + 64 * s + 16 * tq);
                const uint32_t W0[4] = {w0.x, w0.y, w0.z, w0.w}, W1[4] = {w1.x, w1.y, w1.z, w1.w};
                const uint32_t* lut = S.lut + lane;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int m = j >> 1, sh = 16 * (j & 1);
                    const uint32_t a0 = lut[((W0[m] >> sh) & 0xFF) * 32], a2 = lut[((W0[m] >> (sh + 8)) & 0xFF) * 32];
                    const uint32_t a1 = lut[((W1[m] >> sh) & 0xFF) * 32], a3 = lut[((W1[m] >> (sh + 8)) & 0xFF) * 32];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a0, a1, a2, a3, qb[j][nt][0], qb[j][nt][1]);
                }
            } else {   // Q8_0
                const uint8_t* r0 = kr + tk0 * D + 128 * s + 32 * tq;
                const uint8_t* r1 = kr + tk1 * D + 128 * s + 32 * tq;
                const uint4 x0 = *reinterpret_cast<const uint4*>(r0), y0 = *reinterpret_cast<const uint4*>(r0 + 16);
                const uint4 x1 = *reinterpret_cast<const uint4*>(r1), y1 = *reinterpret_cast<const uint4*>(r1 + 16);
                const uint32_t W0[8] = {x0.x, x0.y, x0.z, x0.w, y0.x, y0.y, y0.z, y0.w};
                const uint32_t W1[8] = {x1.x, x1.y, x1.z, x1.w, y1.x, y1.y, y1.z, y1.w};
                const uint16_t* dr = reinterpret_cast<const uint16_t*>(kr + 128 * D);
                const __half2 d0h = __float2half2_rn(h2f(dr[tk0 * (D / 32) + 4 * s + tq]));
                const __half2 d1h = __float2half2_rn(h2f(dr[tk1 * (D / 32) + 4 * s + tq]));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t a0 = as_u(__hmul2(i8pair(W0[j], 0x5140), d0h));
                    const uint32_t a2 = as_u(__hmul2(i8pair(W0[j], 0x7362), d0h));
                    const uint32_t a1 = as_u(__hmul2(i8pair(W1[j], 0x5140), d1h));
                    const uint32_t a3 = as_u(__hmul2(i8pair(W1[j], 0x7362), d1h));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a0, a1, a2, a3, qb[j][nt][0], qb[j][nt][1]);
                }
            }
            // score epilogue: per-row scale / zero point of this slice
            float e0 = 1.f, e1 = 1.f, z0 = 0.f, z1 = 0.f;
            if (kk == KF_KVARN) {
                const uint16_t* sb = reinterpret_cast<const uint16_t*>(ksb);
                e0 = h2f(sb[tk0]); e1 = h2f(sb[tk1]);
                z0 = h2f(sb[128 + tk0]); z1 = h2f(sb[128 + tk1]);
            } else if (kk == KF_TBQ4) {
                const uint16_t* nr = reinterpret_cast<const uint16_t*>(kr + 64 * D);
                e0 = h2f(nr[tk0 * (D / 128) + s]); e1 = h2f(nr[tk1 * (D / 128) + s]);
            }
            float* dst = sxb + (((size_t)(T * TPT + a) * CS + s) * 16) * NQ;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float zq0 = 0.f, zq1 = 0.f;
                if (kk == KF_KVARN) {
                    // sum(q') of queries nt*8 + 2tq (+1) lives in lanes with g = 2tq (+1)
                    zq0 = __shfl_sync(0xffffffffu, sumq[nt], (2 * tq) * 4);
                    zq1 = __shfl_sync(0xffffffffu, sumq[nt], (2 * tq + 1) * 4);
                }
                const int qc = nt * 8 + 2 * tq;
                dst[g * NQ + qc] = e0 * acc[nt][0] + z0 * zq0;
                dst[g * NQ + qc + 1] = e0 * acc[nt][1] + z0 * zq1;
                dst[(g + 8) * NQ + qc] = e1 * acc[nt][2] + z1 * zq0;
                dst[(g + 8) * NQ + qc + 1] = e1 * acc[nt][3] + z1 * zq1;
            }
        }
        if (CS > 1) named_sync(1 + T, CS * 32);
        else __syncwarp();

        // ---------------- full scores, online softmax for the team
        float sv[TPT][NT][4];
        float mt[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mt[nt][0] = mt[nt][1] = -INFINITY;
#pragma unroll
        for (int a = 0; a < TPT; ++a) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int qc = nt * 8 + 2 * tq;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ss = 0; ss < CS; ++ss) {
                    const float* src = sxb + (((size_t)(T * TPT + a) * CS + ss) * 16) * NQ;
                    v[0] += src[g * NQ + qc];
                    v[1] += src[g * NQ + qc + 1];
                    v[2] += src[(g + 8) * NQ + qc];
                    v[3] += src[(g + 8) * NQ + qc + 1];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) sv[a][nt][i] = v[i] * sc;
                mt[nt][0] = fmaxf(mt[nt][0], fmaxf(sv[a][nt][0], sv[a][nt][2]));
                mt[nt][1] = fmaxf(mt[nt][1], fmaxf(sv[a][nt][1], sv[a][nt][3]));
            }
        }
        if (CS > 1) named_sync(1 + T, CS * 32);     // every team warp has read the exchange
        else __syncwarp();
        float alpha[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float m = mt[nt][c];
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                const float mn = fmaxf(m_run[nt][c], m);
                alpha[nt][c] = exp2f(m_run[nt][c] - mn);
                m_run[nt][c] = mn;
            }
        }
        float lsum[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) lsum[nt][0] = lsum[nt][1] = 0.f;
#pragma unroll
        for (int a = 0; a < TPT; ++a)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                sv[a][nt][0] = exp2f(sv[a][nt][0] - m_run[nt][0]);
                sv[a][nt][1] = exp2f(sv[a][nt][1] - m_run[nt][1]);
                sv[a][nt][2] = exp2f(sv[a][nt][2] - m_run[nt][0]);
                sv[a][nt][3] = exp2f(sv[a][nt][3] - m_run[nt][1]);
                lsum[nt][0] += sv[a][nt][0] + sv[a][nt][2];
                lsum[nt][1] += sv[a][nt][1] + sv[a][nt][3];
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float l = lsum[nt][c];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                l_run[nt][c] = l_run[nt][c] * alpha[nt][c] + l;
            }
#pragma unroll
        for (int mtl = 0; mtl < 8; ++mtl)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                O[mtl][nt][0] *= alpha[nt][0];
                O[mtl][nt][1] *= alpha[nt][1];
                O[mtl][nt][2] *= alpha[nt][0];
                O[mtl][nt][3] *= alpha[nt][1];
            }

        // ---------------- P'^T fragments (per tile, per V-scale block) and O += V^T P'^T
        float zs[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) zs[nt][0] = zs[nt][1] = 0.f;
        const int nblk = (vk == KF_Q8 || vk == KF_Q4) ? 4 : 1;
#pragma unroll
        for (int a = 0; a < TPT; ++a) {
            const int tk0 = base - RUN * tq + RUN * (g >> 1) + tok_off(vp, a, g & 1);
            const int tk1 = base - RUN * tq + RUN * (g >> 1) + tok_off(vp, a, 2 + (g & 1));
            uint32_t pb[4][NT][2];
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                if (bb >= nblk) break;
                float f0 = 1.f, f1 = 1.f;
                if (vk == KF_KVARN) {
                    const uint16_t* sb = reinterpret_cast<const uint16_t*>(vsb);
                    f0 = h2f(sb[tk0]); f1 = h2f(sb[tk1]);
                    if (bb == 0) {
                        const float zz0 = h2f(sb[128 + tk0]), zz1 = h2f(sb[128 + tk1]);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            zs[nt][0] += sv[a][nt][0] * zz0 + sv[a][nt][2] * zz1;
                            zs[nt][1] += sv[a][nt][1] * zz0 + sv[a][nt][3] * zz1;
                        }
                    }
                } else if (vk == KF_TBQ4) {
                    const uint16_t* nr = reinterpret_cast<const uint16_t*>(vr + 64 * D);
                    f0 = h2f(nr[tk0 * (D / 128) + s]); f1 = h2f(nr[tk1 * (D / 128) + s]);
                } else {
                    const uint16_t* dr = reinterpret_cast<const uint16_t*>(vr + (vk == KF_Q8 ? 128 : 64) * D);
                    f0 = h2f(dr[tk0 * (D / 32) + 4 * s + bb]);
                    f1 = h2f(dr[tk1 * (D / 32) + 4 * s + bb]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    pb[bb][nt][0] = movtrans(pack_f2(sv[a][nt][0] * f0, sv[a][nt][1] * f0));
                    pb[bb][nt][1] = movtrans(pack_f2(sv[a][nt][2] * f1, sv[a][nt][3] * f1));
                }
            }
#pragma unroll
            for (int mtl = 0; mtl < 8; ++mtl) {
                const int c0 = 128 * s + 16 * mtl + g, c1 = c0 + 8;     // channels of rows g, g+8
                __half2 a0, a1, a2, a3;
                if (vk == KF_KVARN || vk == KF_Q4) {
                    const uint8_t* lo = (vk == KF_KVARN) ? vt : vr;
                    const int cc0 = (vk == KF_KVARN) ? (c0 & 255) : c0, cc1 = (vk == KF_KVARN) ? (c1 & 255) : c1;
                    uint32_t x0, x1;
                    int sh;
                    if (RUN >= 8) {
                        const int wo = (base >> 1) + 4 * (a >> 1);
                        x0 = *reinterpret_cast<const uint32_t*>(lo + cc0 * 64 + wo);
                        x1 = *reinterpret_cast<const uint32_t*>(lo + cc1 * 64 + wo);
                        sh = 8 * (a & 1);
                    } else {
                        x0 = __byte_perm(*reinterpret_cast<const uint16_t*>(lo + cc0 * 64 + (base >> 1)), 0, 0x4140);
                        x1 = __byte_perm(*reinterpret_cast<const uint16_t*>(lo + cc1 * 64 + (base >> 1)), 0, 0x4140);
                        sh = 0;
                    }
                    a0 = nib2(x0, sh); a2 = nib2(x0, sh + 4);
                    a1 = nib2(x1, sh); a3 = nib2(x1, sh + 4);
                    if (vk == KF_KVARN) {
                        if (vbits == 5) {
                            const int bo = base + 8 * (a >> 1) + 2 * (a & 1);    // first position of slot e0
                            const uint32_t hb0 = *reinterpret_cast<const uint32_t*>(lo + 16384 + cc0 * 16 + ((bo >> 3) & ~3));
                            const uint32_t hb1 = *reinterpret_cast<const uint32_t*>(lo + 16384 + cc1 * 16 + ((bo >> 3) & ~3));
                            const int x = bo & 31;
                            const __half2 sixteen = __float2half2_rn(16.f);
                            a0 = __hfma2(bit2(hb0, x), sixteen, a0);
                            a2 = __hfma2(bit2(hb0, x + 1), sixteen, a2);
                            a1 = __hfma2(bit2(hb1, x), sixteen, a1);
                            a3 = __hfma2(bit2(hb1, x + 1), sixteen, a3);
                        }
                        const uint16_t* sb = reinterpret_cast<const uint16_t*>(vsb);
                        const __half2 C0 = __float2half2_rn(h2f(sb[256 + cc0])), C1 = __float2half2_rn(h2f(sb[256 + cc1]));
                        a0 = __hmul2(a0, C0); a2 = __hmul2(a2, C0);
                        a1 = __hmul2(a1, C1); a3 = __hmul2(a3, C1);
                    } else {
                        const __half2 eight = __float2half2_rn(8.f);
                        a0 = __hsub2(a0, eight); a2 = __hsub2(a2, eight);
                        a1 = __hsub2(a1, eight); a3 = __hsub2(a3, eight);
                    }
                } else if (vk == KF_TBQ4) {
                    const int bo = (base >> 1) + 2 * a;
                    const uint16_t y0 = *reinterpret_cast<const uint16_t*>(vr + c0 * 64 + bo);
                    const uint16_t y1 = *reinterpret_cast<const uint16_t*>(vr + c1 * 64 + bo);
                    const uint32_t* lut = S.lut + lane;
                    a0 = as_h2(lut[(y0 & 0xFF) * 32]); a2 = as_h2(lut[(y0 >> 8) * 32]);
                    a1 = as_h2(lut[(y1 & 0xFF) * 32]); a3 = as_h2(lut[(y1 >> 8) * 32]);
                } else {   // Q8_0 V: int8 per position, channel-major rows of 128 bytes
                    const uint32_t y0 = *reinterpret_cast<const uint32_t*>(vr + c0 * 128 + base + 4 * a);
                    const uint32_t y1 = *reinterpret_cast<const uint32_t*>(vr + c1 * 128 + base + 4 * a);
                    a0 = i8pair(y0, 0x5140); a2 = i8pair(y0, 0x7362);
                    a1 = i8pair(y1, 0x5140); a3 = i8pair(y1, 0x7362);
                }
                const int bb = (nblk == 4) ? (mtl >> 1) : 0;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma16816(O[mtl][nt], as_u(a0), as_u(a1), as_u(a2), as_u(a3), pb[bb][nt][0], pb[bb][nt][1]);
            }
        }
        if (vk == KF_KVARN) {
            // O += C_c * sum_t p_t Z_t  (zero point of the V rows, once per group)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float z = zs[nt][c];
                    z += __shfl_xor_sync(0xffffffffu, z, 4);
                    z += __shfl_xor_sync(0xffffffffu, z, 8);
                    z += __shfl_xor_sync(0xffffffffu, z, 16);
                    zs[nt][c] = z;
                }
            const uint16_t* sb = reinterpret_cast<const uint16_t*>(vsb);
#pragma unroll
            for (int mtl = 0; mtl < 8; ++mtl) {
                const float C0 = h2f(sb[256 + ((128 * s + 16 * mtl + g) & 255)]);
                const float C1 = h2f(sb[256 + ((128 * s + 16 * mtl + g + 8) & 255)]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    O[mtl][nt][0] += C0 * zs[nt][0];
                    O[mtl][nt][1] += C0 * zs[nt][1];
                    O[mtl][nt][2] += C1 * zs[nt][0];
                    O[mtl][nt][3] += C1 * zs[nt][1];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&S.empty[sl]));
    }

    // ---- combine the teams (shared memory reuses the stages, all consumed by now)
    named_sync(9, kConsumers * 32);
    float* tstat = reinterpret_cast<float*>(S.stage);                   // [TEAMS][2][NQ]
    float* OT = tstat + C::TEAMS * 2 * NQ;                                // [TEAMS][NQ][D]
    if (s == 0 && g == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                tstat[(T * 2 + 0) * NQ + nt * 8 + 2 * tq + c] = m_run[nt][c];
                tstat[(T * 2 + 1) * NQ + nt * 8 + 2 * tq + c] = l_run[nt][c];
            }
    }
#pragma unroll
    for (int mtl = 0; mtl < 8; ++mtl) {
        const int c0 = 128 * s + 16 * mtl + g;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int qc = nt * 8 + 2 * tq;
            float* ot = OT + (size_t)T * NQ * D;
            ot[qc * D + c0] = O[mtl][nt][0];
            ot[(qc + 1) * D + c0] = O[mtl][nt][1];
            ot[qc * D + c0 + 8] = O[mtl][nt][2];
            ot[(qc + 1) * D + c0 + 8] = O[mtl][nt][3];
        }
    }
    named_sync(9, kConsumers * 32);
    float* part = p.partials + (size_t)item * (2 * NQ + NQ * D);
    float* ofin = OT + (size_t)C::TEAMS * NQ * D;                        // [NQ][D] combined output
    for (int e = threadIdx.x; e < NQ * D; e += kConsumers * 32) {
        const int qi = e / D;
        float m = -INFINITY;
        for (int t = 0; t < C::TEAMS; ++t) m = fmaxf(m, tstat[(t * 2) * NQ + qi]);
        float o = 0.f;
        for (int t = 0; t < C::TEAMS; ++t) {
            const float mt_ = tstat[(t * 2) * NQ + qi];
            if (mt_ != -INFINITY) o += exp2f(mt_ - m) * OT[(size_t)t * NQ * D + e];
        }
        ofin[e] = o;
    }
    if (threadIdx.x < NQ) {
        const int qi = threadIdx.x;
        float m = -INFINITY, l = 0.f;
        for (int t = 0; t < C::TEAMS; ++t) m = fmaxf(m, tstat[(t * 2) * NQ + qi]);
        for (int t = 0; t < C::TEAMS; ++t) {
            const float mt_ = tstat[(t * 2) * NQ + qi];
            if (mt_ != -INFINITY) l += exp2f(mt_ - m) * tstat[(t * 2 + 1) * NQ + qi];
        }
        part[qi] = m;
        part[NQ + qi] = l;
    }
    named_sync(9, kConsumers * 32);
    rotate_rows_c(ofin, NQ, D, L.rot, true);
    float4* po = reinterpret_cast<float4*>(part + 2 * NQ);
    const float4* q4 = reinterpret_cast<const float4*>(ofin);
    for (int e = threadIdx.x; e < NQ * D / 4; e += kConsumers * 32) po[e] = q4[e];
}

template <int D, int NQ>
size_t body_fixed_smem(bool lut) {
    using C = BodyCfg<D, NQ>;
    return 128 + (lut ? kLutBytes : 0) + (size_t)C::Q_BYTES + (size_t)C::SX_FLOATS * 4;
}

template <int D, int NQ>
int launch_body_t(const Layout& L, const AttnParams& p, int n_body, cudaStream_t st) {
    const uint32_t recK = (uint32_t)L.rec_bytes[0], recV = (uint32_t)L.rec_bytes[1];
    const size_t v_off = (recK + 127u) & ~127u;
    const size_t stage = (v_off + recV + 127u) & ~127u;
    const bool lut = (L.fmt[0] == KVQ_TBQ4) || (L.fmt[1] == KVQ_TBQ4);
    const size_t fixed = body_fixed_smem<D, NQ>(lut);
    const size_t budget = 227 * 1024;
    int nst = (int)((budget - fixed) / stage);
    if (nst > 4) nst = 4;
    if (nst < 2) return (int)cudaErrorInvalidConfiguration;
    // the team-combine area reuses the stages: it must fit there
    using C = BodyCfg<D, NQ>;
    const size_t combine = ((size_t)C::TEAMS * 2 * NQ + (size_t)(C::TEAMS + 1) * NQ * D) * 4;
    if (combine > (size_t)nst * stage) return (int)cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)nst * stage + fixed;
    cudaFuncSetAttribute(decode_body_kernel<D, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_body_kernel<D, NQ><<<n_body, kBodyThreads, smem, st>>>(L, p, nst);
    return (int)cudaGetLastError();
}

template <int D, int NQ>
int ctas_per_sm_t(const Layout& L) {
    const uint32_t recK = (uint32_t)L.rec_bytes[0], recV = (uint32_t)L.rec_bytes[1];
    const size_t stage = ((((recK + 127u) & ~127u) + recV + 127u) & ~127u);
    const bool lut = (L.fmt[0] == KVQ_TBQ4) || (L.fmt[1] == KVQ_TBQ4);
    const size_t fixed = body_fixed_smem<D, NQ>(lut);
    const size_t budget = 227 * 1024;
    int nst = (int)((budget - fixed) / stage);
    if (nst > 4) nst = 4;
    return nst >= 2 ? 1 : 0;
}

}  // namespace

int body_ctas_per_sm(const Layout& L) {
    if (L.NQ == 8) {
        if (L.D == 128) return ctas_per_sm_t<128, 8>(L);
        if (L.D == 256) return ctas_per_sm_t<256, 8>(L);
        if (L.D == 512) return ctas_per_sm_t<512, 8>(L);
    } else {
        if (L.D == 128) return ctas_per_sm_t<128, 16>(L);
        if (L.D == 256) return ctas_per_sm_t<256, 16>(L);
        if (L.D == 512) return ctas_per_sm_t<512, 16>(L);
    }
    return 0;
}

int upload_tables_body(const FormatTables& t) {
    return (int)cudaMemcpyToSymbol(c_tab, &t, sizeof(FormatTables));
}

// Launches the body kernel over the last n_body work items of p (the body items).
int launch_decode_body(const Layout& L, const AttnParams& p, int n_body, void* stream) {
    if (n_body <= 0) return 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (L.NQ == 8) {
        if (L.D == 128) return launch_body_t<128, 8>(L, p, n_body, s);
        if (L.D == 256) return launch_body_t<256, 8>(L, p, n_body, s);
        if (L.D == 512) return launch_body_t<512, 8>(L, p, n_body, s);
    } else {
        if (L.D == 128) return launch_body_t<128, 16>(L, p, n_body, s);
        if (L.D == 256) return launch_body_t<256, 16>(L, p, n_body, s);
        if (L.D == 512) return launch_body_t<512, 16>(L, p, n_body, s);
    }
    return (int)cudaErrorInvalidValue;
}

}  // namespace kvq
