// Decode attention over the unsealed regions: the tq6_0 ring span (rotated domain) and the
// 16-bit rows of the sink, the exact tail and an exact journal (original domain). bf16 rows use
// the bf16 mma with the query and P' each split into bf16 high and low parts (16 significant bits).
//
// One CTA of 8 warps per region work item (sequence, KV head, run of positions inside one
// region), in runs of up to 128 positions; the fused decode kernel (kernels_body.cu) runs these
// items after its body items. Thread 0 streams each run into shared memory with cp.async.bulk:
// one copy per contiguous slot range of the K rows, V rows and tq6_0 scale rows (many small
// copies per run cost far more TMA time than a few large ones). The warps consume each run like
// the body items:
//   1. scores: warp w takes positions [16w, 16w + 16) and all D channels. tq6_0 K rows are
//      decoded straight into mma.sync m16n8k16 A fragments (6-bit code c: nibble in mantissa
//      bits 4-7 and the two high bits in bits 8-9 of a half with exponent 6, i.e. 64 + c);
//      fp16 K rows are the A fragments as they stand. Positions past the run's end score -inf.
//   2. group maximum, p = 2^(s - m), running sums, P' = p x (tq6_0 value scale of the block);
//      movmatrix gives the B fragments of step 3 (one 8-byte store per lane).
//   3. values: warp w takes channels [wD/8, (w+1)D/8) (fp16 rows come in runs of 48 positions
//      beside a ring, 32 at head_dim 512; warps past the run skip step 1). The rows are token-major, so the A
//      fragments of V^T come from transposes: ldmatrix.trans of the fp16 rows; for the ring,
//      tq6_0 codes decoded in registers as 8 x 8 tiles (positions x channel pairs) and
//      transposed by movmatrix (head_dim 256), or decoded into a small per-warp buffer that
//      ldmatrix.trans reads back (head_dim 128); either way the fragment rows hold the channels
//      in a fixed permutation that the partial's write undoes. An all-ones mma gives sum_t P'_t,
//      which removes the code offset 96 (64 + the tq6_0 centre 32) once per run.
// The partial (m, l, o) of a ring item is rotated back to the original domain; the merge
// kernel (kernels_attn.cu) combines all partials of a (sequence, KV head) under one softmax.
#pragma once
#include <cuda_bf16.h>
#include "stream_common.cuh"
#include "append_row.cuh"

namespace kvq {
namespace {

// The fused decode step's append of the newest position (128 threads per row, see
// codec::append_row), out of line: cold code kept out of the decode loops' instruction stream.
__device__ __noinline__ void append_newest(const Layout& L, const void* pool, int64_t unit, int w, int pos,
                                           const uint16_t* src, int tid, uint8_t* cs) {
    codec::append_row(L, pool, unit, w, pos, src, true, tid, 128, cs);
}

template <int D, int NQ>
struct RGeo {
    static constexpr int NT = NQ / 8;
    static constexpr int KS = D / 16;
    static constexpr int MT = D / 128;
    static constexpr int NB = D / 128;                                  // tq6_0 blocks per row
    static constexpr int CODE_ROW = NB * 96;                            // tq6_0 code row bytes
    static constexpr int CLD = CODE_ROW;                                // smem row stride (dense)
    static constexpr int SC_BYTES = (128 * NB * 2 + 15) & ~15;         // scale rows of a run
    static constexpr int TQ_HALF = 128 * CLD + SC_BYTES;                // K (or V) part of a ring stage
    static constexpr int TQ_STAGE = 2 * TQ_HALF;
    static constexpr int FLD = 2 * D;                                   // fp16 row stride (dense)
    // head_dim 512 takes 16-bit rows only (no tq6_0 ring; the host routes rings at 512 to the
    // generic kernel); its staging area is two 64 KB fp16 stages (one CTA per SM). With a ring the
    // staging area is two tq6_0 stages, and the fp16 runs are sized so that two of them fit too
    // (thread 0 refills a stage only after the next run's first barrier: two stages at least).
    static constexpr bool RING = D <= 256;
    static constexpr int RUNF = !RING ? 16384 / D : (TQ_STAGE / (4 * D)) & ~15;   // fp16 rows per run
    static constexpr int F_HALF = RUNF * FLD;
    static constexpr int F_STAGE = 2 * F_HALF;
    static constexpr int AREA = !RING ? 2 * F_STAGE : 2 * TQ_STAGE;
    static_assert(RUNF >= 16 && RUNF <= 128 && AREA >= 2 * F_STAGE, "two fp16 stages of whole k-steps");
    static constexpr int QB_BYTES = NT * KS * 256;                      // one fragment set
    static constexpr int PC = (RING && NB > 2) ? NB : 2;                // P' copies (bf16 rows: hi, lo)
    static constexpr int P_BYTES = PC * 8 * NT * 256;
    static_assert(P_BYTES >= 2 * D, "the P' area stages the codes of a fused append");
    static constexpr int RED_FLOATS = 2 * NQ * 8 + 2 * NQ;
    // tq6_0 values: per-warp buffer of decoded rows (ROWS positions x the warp's D/8 channels,
    // fp16, padded rows) read back transposed by ldmatrix
    static constexpr int CPW = D / 8, WPP = CPW / 8, VROWS = 32 / WPP, VRS = CPW * 2 + 16;
    static constexpr int VB_BYTES = VROWS * VRS;
    // shared memory: one query-fragment set, a second one for layouts with bf16 rows
    static constexpr int smem(bool bf16_rows) {
        return AREA + 128 + (bf16_rows ? 2 : 1) * QB_BYTES + P_BYTES + RED_FLOATS * 4 + kConsumers * VB_BYTES;
    }
    static constexpr int NTASK = NQ * D / 8;
    static constexpr int TPT = (NTASK + kCT - 1) / kCT;
};

// The two high bits of 8 tq6_0 codes (16 bits, code i at bits 2i) spread for hi2_at: codes
// 0..3 at bits 0-7, codes 4..7 at bits 16-23.
__device__ __forceinline__ uint32_t hi2_spread(uint32_t h16) { return (h16 & 0xFFu) | ((h16 & 0xFF00u) << 8); }
// Adds the high bits of codes x and x+4 (from hi2_spread) to a nib64 pair: mantissa bits 8-9.
template <int X>
__device__ __forceinline__ uint32_t hi2_at(uint32_t raw, uint32_t u) { return ((u << (8 - 2 * X)) & 0x03000300u) | raw; }
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// A pair of floats as bf16 (round to nearest even): the high part and the remainder, so that
// hi + lo carries 16 significant bits.
__device__ __forceinline__ void split_bf2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// One region work item, run by a CTA of 8 warps on the dynamic shared memory `smem`; s_abort is
// the CTA's abort flag (a __shared__ int). RK: the region kinds the layout can hold (bit 0: a
// tq6_0 ring, bit 1: bf16 rows); an instance compiles only their readers. ROT: the layout's
// rotation (that of the ring's rows).
template <int D, int NQ, int RK, int ROT>
__device__ __forceinline__ void region_item(const Layout& L, const AttnParams& p, const int item, uint8_t* smem,
                                            int& s_abort) {
    using Gm = RGeo<D, NQ>;
    constexpr int NT = Gm::NT, KS = Gm::KS, MT = Gm::MT, NB = Gm::NB, TPT = Gm::TPT;
    constexpr int CLD = Gm::CLD, FLD = Gm::FLD;

    // ---- work item (same enumeration as the generic region kernel)
    int b = 0;
    while (b + 1 < p.n_seq && p.seq[b + 1].first_item <= item) ++b;
    const SeqSpan& sp = p.seq[b];
    const int local = item - sp.first_item;
    const int h = local / sp.items_per_head;
    int cidx = local % sp.items_per_head, r = 0;
    while (r < 3 && cidx >= sp.nchunk[r]) { cidx -= sp.nchunk[r]; ++r; }
    const int kind = sp.kind[r];
    const int ck = (kind == RK_RING) ? p.ring_chunk : p.chunk;
    const int t0 = sp.lo[r] + cidx * ck;
    const int t1 = min(t0 + ck, sp.hi[r]);
    const bool ring = Gm::RING && (RK & 1) && (kind == RK_RING);
    // bf16 exact rows: bf16 mma, the query and P' each split into bf16 high and low parts
    const bool bf = (RK & 2) && !ring && kind != RK_SINK && ((kind == RK_TAIL ? L.tail_fmt : L.journal) == KVQ_BF16);
    const int RUN = ring ? 128 : Gm::RUNF;                // positions per run
    const int nrun = (t1 - t0 + RUN - 1) / RUN;
    const int64_t unit = L.unit(p.layer, sp.slot, h);
    uint32_t* status = status_word(L, p.pool);

    const uint32_t stage_bytes = ring ? Gm::TQ_STAGE : Gm::F_STAGE;
    const uint32_t half_bytes = ring ? Gm::TQ_HALF : Gm::F_HALF;
    const int nst = min(4, Gm::AREA / (int)stage_bytes);
    // a ring at head_dim 512 is not routed here, nor to an instance without the ring reader: refuse
    if (nst < 2 || ((!Gm::RING || !(RK & 1)) && kind == RK_RING)) {
        grid_dep_wait();
        if (threadIdx.x == 0) atomicOr(status_word(L, p.pool), 4u);
        return;
    }
    uint8_t* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Gm::AREA);
    uint8_t* cur = smem + Gm::AREA + 128;
    const bool has_bf = (RK & 2) && ((L.tail_fmt == KVQ_BF16) || (L.journal == KVQ_BF16));
    uint32_t* qb = reinterpret_cast<uint32_t*>(cur);      cur += (has_bf ? 2 : 1) * Gm::QB_BYTES;   // bf16: hi, lo
    uint32_t* pbuf = reinterpret_cast<uint32_t*>(cur);    cur += Gm::P_BYTES;
    float* red = reinterpret_cast<float*>(cur);           // [NQ][warp] maxima, then sums; m at 2 NQ 8
    cur += Gm::RED_FLOATS * 4;
    uint8_t* vbuf = cur;                                  // [warp][VROWS][VRS] decoded tq6_0 values

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // thread 0 streams the runs: run i into stage i % nst, issued once stage i % nst is free
    // (the first barrier of run i - nst + 1 follows every read of run i - nst)
    int isl = 0;                                          // stage of the next issue (thread 0): i % nst
    auto issue = [&](int i) {
        const int sl = isl;
        isl = (isl + 1 == nst) ? 0 : isl + 1;
        const int pc = t0 + RUN * i, n = min(RUN, t1 - pc);
        uint8_t* st = stages + (size_t)sl * stage_bytes;
        const uint32_t fb = su32(&full[sl]);
        // contiguous slot runs: one copy each (a run of the ring never wraps; the tail and an
        // exact journal wrap at most once)
        {
            if (ring) {
                mbar_expect_tx(fb, 2u * (n * Gm::CODE_ROW + Gm::SC_BYTES));
                for (int w = 0; w < 2; ++w) {
                    uint8_t* dst = st + w * half_bytes;
                    const int s0 = journal_slot(L, pc);
                    bulk_g2s(su32(dst), jcode_row(L, p.pool, w, unit, s0), n * Gm::CODE_ROW, fb);
                    bulk_g2s(su32(dst + 128 * CLD), jscale_row(L, p.pool, w, unit, s0), Gm::SC_BYTES, fb);
                }
            } else {
                mbar_expect_tx(fb, 2u * n * 2 * D);
                // a fused decode step's newest position (the last row of the sequence) comes
                // from the caller's input row (fp16, which the host checks)
                const bool newest = (p.knew != nullptr) && (pc + n == sp.n_tok);
                for (int w = 0; w < 2; ++w) {
                    uint8_t* dst = st + w * half_bytes;
                    const int ncache = newest ? n - 1 : n;
                    if (newest)
                        bulk_g2s(su32(dst + ncache * FLD), (w ? p.vnew : p.knew) + ((int64_t)b * L.H + h) * D, 2 * D, fb);
                    int done = 0;
                    while (done < ncache) {
                        const int pos = pc + done;
                        const uint16_t* src;
                        int cnt;
                        if (kind == RK_SINK) {
                            src = sink_row(L, p.pool, w, unit, pos);
                            cnt = ncache - done;
                        } else if (kind == RK_TAIL) {
                            const int sl0 = pos % L.T;
                            src = tail_row(L, p.pool, w, unit, sl0);
                            cnt = min(ncache - done, L.T - sl0);
                        } else {
                            const int sl0 = journal_slot(L, pos);
                            src = jexact_row(L, p.pool, w, unit, sl0);
                            cnt = min(ncache - done, L.R - sl0);
                        }
                        bulk_g2s(su32(dst + done * FLD), src, cnt * 2 * D, fb);
                        done += cnt;
                    }
                }
            }
        }
    };
    // the query rows of the head (G x D fp16, contiguous) land in the fragment area first: the
    // set-up waits on them (full[4]) while the first runs stream in behind them
    const int G = L.G;
    const uint16_t* qsrc = p.q + ((int64_t)b * L.Hq + (int64_t)h * G) * D;
    const uint32_t qbar = su32(&full[4]);
    int issued = 0;
    if (threadIdx.x == 0) {   // barriers first: no global memory is touched before the wait
        s_abort = 0;
        for (int i = 0; i < 5; ++i) mbar_init(su32(&full[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (!p.early) grid_dep_wait();   // the launch ahead (programmatic serialization) has completed
    if (threadIdx.x == 0) {
        mbar_expect_tx(qbar, (uint32_t)(G * D * 2));
        bulk_g2s(su32(qb), qsrc, (uint32_t)(G * D * 2), qbar);
        for (; issued < min(nst, nrun); ++issued) issue(issued);
    }
    __syncthreads();
    if (p.knew != nullptr && t1 == sp.n_tok && sp.body_per_head == 0) {
        // fused decode step, sequence without body items: the item that holds the newest
        // position appends it to the cache (threads 0-127 the K row, 128-255 the V row; codes
        // staged in the P' area, unused yet). Nothing in this launch reads the slots written:
        // the newest row is read from the input above, and its ring slot holds no position of
        // the ring span (the journal never holds more than R positions)
        const int w = threadIdx.x >> 7;
        append_newest(L, p.pool, unit, w, sp.n_tok - 1, (w ? p.vnew : p.knew) + ((int64_t)b * L.H + h) * D,
                      threadIdx.x & 127, reinterpret_cast<uint8_t*>(pbuf) + w * D);
    }

    // ================================================================== consumers: set-up
    const int g = lane >> 2, tq = lane & 3;
    __half* qr = reinterpret_cast<__half*>(qb);           // query rows, fp16 [NQ][D], rotated in place
    mbar_wait(qbar, 0, status, &s_abort);
    {
        const uint16_t* q = reinterpret_cast<const uint16_t*>(qr);
        const int rot = ring ? ROT : (int)ROT_NONE;
        if (rot == ROT_HAD256) {
            if constexpr (D >= 256) {
                for (int u = warp; u < NQ * (D / 256); u += kConsumers) {
                    const int rr = u / (D / 256), c0 = (u % (D / 256)) * 256;
                    float v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[k] = (rr < G) ? h2f(q[rr * D + c0 + lane + 32 * k]) : 0.f;
                    warp_rotate<8>(v, lane, rot);
#pragma unroll
                    for (int k = 0; k < 8; ++k) qr[rr * D + c0 + lane + 32 * k] = __float2half_rn(v[k]);
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
                for (int k = 0; k < 4; ++k) qr[rr * D + c0 + lane + 32 * k] = __float2half_rn(v[k]);
            }
        }
    }
    csync();
    // Query fragments. tq6_0 K: thread quad tq holds channels [32 tq, 32 tq + 32) of every
    // 128-channel block, k-step pairs (x, x+4) of 8-channel words. fp16 K: thread quad tq holds
    // the 16-byte chunks 4i + tq of the row, k-steps 2i and 2i + 1 in natural pairs.
    uint2 qe0[TPT], qe1[TPT], ql0[TPT], ql1[TPT];
    int qidx[TPT];
#pragma unroll
    for (int k = 0; k < TPT; ++k) {
        const int t = threadIdx.x + kCT * k;
        qidx[k] = -1;
        if (t < Gm::NTASK) {
            // lanes of a warp take the 32 entries (query, quad) of one k-step pair
            const int ln = t & 31, rest = t >> 5;
            const int tq_ = ln & 3, nt_ = rest % NT, jb = rest / NT;
            const int qi = nt_ * 8 + (ln >> 2);
            int u, j0;
            if (ring) {   // 128-channel blocks, quad tq holds channels [32 tq, 32 tq + 32) of each
                const int bb = jb / 4, m = jb % 4;
                u = bb * 16 + tq_ * 4 + m;
                j0 = bb * 8 + 2 * m;
            } else {      // chunk 4 jb + tq
                u = 4 * jb + tq_;
                j0 = 2 * jb;
            }
            qidx[k] = (((qi >> 3) * KS + j0) * 8 + (qi & 7)) * 4 + tq_;
            const uint4 x = *reinterpret_cast<const uint4*>(qr + qi * D + 8 * u);
            if (ring) {
                qe0[k] = make_uint2(__byte_perm(x.x, x.z, 0x5410), __byte_perm(x.x, x.z, 0x7632));
                qe1[k] = make_uint2(__byte_perm(x.y, x.w, 0x5410), __byte_perm(x.y, x.w, 0x7632));
            } else if (bf) {
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __half22float2(as_h2(xs[i]));
                    split_bf2(f.x, f.y, hi[i], lo[i]);
                }
                qe0[k] = make_uint2(hi[0], hi[1]);
                qe1[k] = make_uint2(hi[2], hi[3]);
                ql0[k] = make_uint2(lo[0], lo[1]);
                ql1[k] = make_uint2(lo[2], lo[3]);
            } else {
                qe0[k] = make_uint2(x.x, x.y);
                qe1[k] = make_uint2(x.z, x.w);
            }
        }
    }
    csync();
#pragma unroll
    for (int k = 0; k < TPT; ++k) {
        if (qidx[k] < 0) continue;
        uint2* e = reinterpret_cast<uint2*>(qb) + qidx[k];
        e[0] = qe0[k];
        e[32] = qe1[k];
        if (bf) {
            e[Gm::QB_BYTES / 8] = ql0[k];
            e[Gm::QB_BYTES / 8 + 32] = ql1[k];
        }
    }
    csync();
    const uint2* qb2 = reinterpret_cast<const uint2*>(qb);
    const uint2* pb2 = reinterpret_cast<const uint2*>(pbuf);
    constexpr uint32_t ONE2 = 0x3C003C00u;
    // ring: sum of the query fragments per 128-channel block (offset 96 of the raw codes)
    float zk[NB][NT][2];
#pragma unroll
    for (int bk = 0; bk < NB; ++bk)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            zk[bk][nt][0] = zk[bk][nt][1] = 0.f;
            if (ring) {
                float a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const uint2 bq = qb2[((nt * KS + bk * 8 + jj) * 8 + g) * 4 + tq];
                    mma16816(a1, ONE2, ONE2, ONE2, ONE2, bq.x, bq.y);
                }
                zk[bk][nt][0] = a1[0];
                zk[bk][nt][1] = a1[1];
            }
        }

    const int r0 = 16 * warp + g, r1 = r0 + 8;            // this thread's score rows (positions in the run)
    const int vw = (warp * (D / 8)) >> 7;                 // tq6_0 block of this warp's value channels
    const float sc = L.scale * kLog2e;
    float m_run[NT][2], l_part[NT][2];
    float O[MT][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_part[nt][0] = l_part[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) O[mt][nt][0] = O[mt][nt][1] = O[mt][nt][2] = O[mt][nt][3] = 0.f;
    }

    // the stage of run gi (gi % nst) and its barrier phase ((gi / nst) & 1), stepped per run
    int sl = 0;
    uint32_t phase = 0;
    for (int gi = 0; gi < nrun; ++gi, sl = (sl + 1 == nst) ? 0 : sl + 1, phase ^= (sl == 0)) {
        mbar_wait(su32(&full[sl]), phase, status, &s_abort);
        const int n = min(RUN, t1 - (t0 + RUN * gi));
        uint8_t* kr = stages + (size_t)sl * stage_bytes;
        uint8_t* vr = kr + half_bytes;
        if (bf && p.knew != nullptr && t0 + RUN * gi + n == sp.n_tok) {
            // fused decode step, bf16 rows: the newest row came from the caller's fp16 input;
            // round it to bf16, the value the cache stores, before any warp reads it
            for (int e = threadIdx.x; e < 2 * D; e += kCT) {
                uint16_t* x = reinterpret_cast<uint16_t*>((e < D ? kr : vr) + (n - 1) * FLD) + (e % D);
                *x = f2bf_bits(h2f(*x));
            }
            csync();
        }
        if (!ring && n < RUN) {   // rows past the run's end: zeros, so 0 x row stays 0 in P.V
            for (int e = threadIdx.x; e < (RUN - n) * (2 * D / 16); e += kCT) {
                const int rr = n + e / (2 * D / 16), u = e % (2 * D / 16);
                *reinterpret_cast<uint4*>(vr + rr * FLD + 16 * u) = make_uint4(0, 0, 0, 0);
            }
        }

        // ---------------- step 1: scores of rows r0, r1
        float s4[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) s4[nt][0] = s4[nt][1] = s4[nt][2] = s4[nt][3] = 0.f;
        if (ring) {
            const uint16_t* ksc = reinterpret_cast<const uint16_t*>(kr + 128 * CLD);
#pragma unroll
            for (int bk = 0; bk < NB; ++bk) {
                float acc[2][NT][4];   // two mma chains, by k-step parity
#pragma unroll
                for (int ch = 0; ch < 2; ++ch)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) acc[ch][nt][0] = acc[ch][nt][1] = acc[ch][nt][2] = acc[ch][nt][3] = 0.f;
                const uint8_t* row0 = kr + r0 * CLD + 96 * bk;
                const uint8_t* row1 = kr + r1 * CLD + 96 * bk;
                const uint4 w0 = *reinterpret_cast<const uint4*>(row0 + 16 * tq);
                const uint4 w1 = *reinterpret_cast<const uint4*>(row1 + 16 * tq);
                const uint2 h0 = *reinterpret_cast<const uint2*>(row0 + 64 + 8 * tq);
                const uint2 h1 = *reinterpret_cast<const uint2*>(row1 + 64 + 8 * tq);
                const uint32_t W0[4] = {w0.x, w0.y, w0.z, w0.w}, W1[4] = {w1.x, w1.y, w1.z, w1.w};
                const uint32_t H0[2] = {h0.x, h0.y}, H1[2] = {h1.x, h1.y};
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int m = jj >> 1;
                    const uint32_t u0 = hi2_spread((H0[m >> 1] >> (16 * (m & 1))) & 0xFFFFu);
                    const uint32_t u1 = hi2_spread((H1[m >> 1] >> (16 * (m & 1))) & 0xFFFFu);
                    uint32_t a0, a1, a2, a3;
                    if (jj & 1) {
                        a0 = hi2_at<2>(nib64(W0[m], 2), u0); a2 = hi2_at<3>(nib64(W0[m], 3), u0);
                        a1 = hi2_at<2>(nib64(W1[m], 2), u1); a3 = hi2_at<3>(nib64(W1[m], 3), u1);
                    } else {
                        a0 = hi2_at<0>(nib64(W0[m], 0), u0); a2 = hi2_at<1>(nib64(W0[m], 1), u0);
                        a1 = hi2_at<0>(nib64(W1[m], 0), u1); a3 = hi2_at<1>(nib64(W1[m], 1), u1);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint2 bq = qb2[((nt * KS + bk * 8 + jj) * 8 + g) * 4 + tq];
                        mma16816(acc[jj & 1][nt], a0, a1, a2, a3, bq.x, bq.y);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[0][nt][i] += acc[1][nt][i];
                const float e0 = h2f(ksc[r0 * NB + bk]), e1 = h2f(ksc[r1 * NB + bk]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float o0 = 96.f * zk[bk][nt][0], o1 = 96.f * zk[bk][nt][1];
                    s4[nt][0] += e0 * (acc[0][nt][0] - o0);
                    s4[nt][1] += e0 * (acc[0][nt][1] - o1);
                    s4[nt][2] += e1 * (acc[0][nt][2] - o0);
                    s4[nt][3] += e1 * (acc[0][nt][3] - o1);
                }
            }
        } else if (16 * warp < RUN) {
            // 16-byte chunk 4i + tq of rows r0, r1; odd rows load chunk pairs in the other order;
            // a second mma chain (sb) takes the odd k-steps
            float sb[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) sb[nt][0] = sb[nt][1] = sb[nt][2] = sb[nt][3] = 0.f;
            const int odd = g & 1;
#pragma unroll
            for (int i2 = 0; i2 < D / 64; ++i2) {
                uint4 c0a = *reinterpret_cast<const uint4*>(kr + r0 * FLD + 16 * (4 * (2 * i2 + odd) + tq));
                uint4 c0b = *reinterpret_cast<const uint4*>(kr + r0 * FLD + 16 * (4 * (2 * i2 + 1 - odd) + tq));
                uint4 c1a = *reinterpret_cast<const uint4*>(kr + r1 * FLD + 16 * (4 * (2 * i2 + odd) + tq));
                uint4 c1b = *reinterpret_cast<const uint4*>(kr + r1 * FLD + 16 * (4 * (2 * i2 + 1 - odd) + tq));
                if (odd) {
                    const uint4 t = c0a; c0a = c0b; c0b = t;
                    const uint4 u = c1a; c1a = c1b; c1b = u;
                }
                const uint32_t A0[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
                const uint32_t A1[8] = {c1a.x, c1a.y, c1a.z, c1a.w, c1b.x, c1b.y, c1b.z, c1b.w};
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = 4 * i2 + jj;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int qix = ((nt * KS + j) * 8 + g) * 4 + tq;
                        const uint2 bq = qb2[qix];
                        if (bf) {   // high part in s4, low part in sb
                            const uint2 bl = qb2[Gm::QB_BYTES / 8 + qix];
                            mma_bf16(s4[nt], A0[2 * jj], A1[2 * jj], A0[2 * jj + 1], A1[2 * jj + 1], bq.x, bq.y);
                            mma_bf16(sb[nt], A0[2 * jj], A1[2 * jj], A0[2 * jj + 1], A1[2 * jj + 1], bl.x, bl.y);
                        } else {
                            mma16816((jj & 1) ? sb[nt] : s4[nt], A0[2 * jj], A1[2 * jj], A0[2 * jj + 1],
                                     A1[2 * jj + 1], bq.x, bq.y);
                        }
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s4[nt][i] += sb[nt][i];
        }
        const bool v0 = r0 < n, v1 = r1 < n;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            s4[nt][0] = v0 ? s4[nt][0] * sc : -INFINITY;
            s4[nt][1] = v0 ? s4[nt][1] * sc : -INFINITY;
            s4[nt][2] = v1 ? s4[nt][2] * sc : -INFINITY;
            s4[nt][3] = v1 ? s4[nt][3] * sc : -INFINITY;
            float mx0 = fmaxf(s4[nt][0], s4[nt][2]), mx1 = fmaxf(s4[nt][1], s4[nt][3]);
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            if (g == 0) {
                red[(nt * 8 + 2 * tq) * 8 + warp] = mx0;
                red[(nt * 8 + 2 * tq + 1) * 8 + warp] = mx1;
            }
        }
        csync();
        if (threadIdx.x == 0 && gi >= 1 && issued < nrun) issue(issued++);

        // ---------------- step 2: group maximum, p, running sums, P' fragments
        float al[NT][2], pr[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float4* r4 = reinterpret_cast<const float4*>(red + (nt * 8 + 2 * tq + c) * 8);
                const float4 x = r4[0], y = r4[1];
                const float gm = fmaxf(fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)), fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
                const float mn = fmaxf(m_run[nt][c], gm);
                al[nt][c] = exp2f(m_run[nt][c] - mn);
                m_run[nt][c] = mn;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) pr[nt][i] = exp2f(s4[nt][i] - m_run[nt][i & 1]);
#pragma unroll
            for (int c = 0; c < 2; ++c) l_part[nt][c] = al[nt][c] * l_part[nt][c] + pr[nt][c] + pr[nt][c + 2];
        }
        const uint16_t* vsc = reinterpret_cast<const uint16_t*>(vr + 128 * CLD);
        if (bf) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint32_t h0, l0, h1, l1;
                split_bf2(v0 ? pr[nt][0] : 0.f, v0 ? pr[nt][1] : 0.f, h0, l0);
                split_bf2(v1 ? pr[nt][2] : 0.f, v1 ? pr[nt][3] : 0.f, h1, l1);
                reinterpret_cast<uint2*>(pbuf)[((0 * 8 + warp) * NT + nt) * 32 + lane] = make_uint2(movtrans(h0), movtrans(h1));
                reinterpret_cast<uint2*>(pbuf)[((1 * 8 + warp) * NT + nt) * 32 + lane] = make_uint2(movtrans(l0), movtrans(l1));
            }
        }
#pragma unroll
        for (int v = 0; v < NB; ++v) {
            if (!ring && (bf || v > 0)) break;
            const float f0 = ring ? h2f(vsc[r0 * NB + v]) : 1.f, f1 = ring ? h2f(vsc[r1 * NB + v]) : 1.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t P0 = v0 ? pack_f2(pr[nt][0] * f0, pr[nt][1] * f0) : 0u;
                const uint32_t P1 = v1 ? pack_f2(pr[nt][2] * f1, pr[nt][3] * f1) : 0u;
                reinterpret_cast<uint2*>(pbuf)[((v * 8 + warp) * NT + nt) * 32 + lane] =
                    make_uint2(movtrans(P0), movtrans(P1));
            }
        }
        csync();

        // ---------------- step 3: O^T = alpha O^T + V^T P'^T for this warp's channels
        const int pv = ring ? vw : 0;
        // k-steps outer, m-tiles inner: the m-tiles' mma chains interleave (one m-tile splits its
        // chain by k-step parity); the all-ones mma is shared by the m-tiles
        constexpr int C3 = (MT == 1) ? 2 : 1;
        float acc[MT][C3][NT][4], a1s[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int i = 0; i < 4; ++i) a1s[nt][i] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int ch = 0; ch < C3; ++ch)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[mt][ch][nt][i] = 0.f;
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if (16 * kk >= RUN) break;
            uint2 bp[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                bp[nt] = pb2[((pv * 8 + kk) * NT + nt) * 32 + lane];
                if (ring) mma16816(a1s[nt], ONE2, ONE2, ONE2, ONE2, bp[nt].x, bp[nt].y);
            }
            // tq6_0 values: this warp decodes VROWS positions x its D/8 channels per fill (a full
            // word per lane: nibble pairs and high bits in a few operations) into its buffer, and
            // ldmatrix.trans reads the A fragments of V^T back (rows hold channels 0,4,1,5,2,6,3,7)
            uint32_t ar[MT][4];
            if (ring && Gm::CPW == 32) {
                // D 256: no staging buffer. Thread (g, tq) decodes channels 8 tq .. 8 tq + 7 of the
                // warp's 32 (register k: channels k and k + 4) of positions g and 8 + g of the k-step;
                // register k over the 8 positions of an octet is an 8 x 8 tile (rows positions,
                // column pairs tq) that movmatrix turns into 8 rows of V^T: row g' = channel
                // 8 (g' >> 1) + k + 4 (g' & 1). m-tile mt takes tiles 2 mt (rows 0-7) and 2 mt + 1.
                const int cw = warp * 32 + 8 * tq;
                uint32_t tl[2][4];
#pragma unroll
                for (int o = 0; o < 2; ++o) {
                    const uint8_t* rowp = vr + (16 * kk + 8 * o + g) * CLD + 96 * (cw >> 7);
                    const uint32_t wq = *reinterpret_cast<const uint32_t*>(rowp + ((cw & 127) >> 1));
                    const uint32_t u = hi2_spread(*reinterpret_cast<const uint16_t*>(rowp + 64 + ((cw & 127) >> 2)));
                    tl[o][0] = movtrans(hi2_at<0>(nib64(wq, 0), u));
                    tl[o][1] = movtrans(hi2_at<1>(nib64(wq, 1), u));
                    tl[o][2] = movtrans(hi2_at<2>(nib64(wq, 2), u));
                    tl[o][3] = movtrans(hi2_at<3>(nib64(wq, 3), u));
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    ar[mt][0] = tl[0][(2 * mt) & 3];
                    ar[mt][1] = tl[0][(2 * mt + 1) & 3];
                    ar[mt][2] = tl[1][(2 * mt) & 3];
                    ar[mt][3] = tl[1][(2 * mt + 1) & 3];
                }
            } else if (ring) {
                constexpr int WPP = Gm::WPP, VROWS = Gm::VROWS, VRS = Gm::VRS, NF = 16 / Gm::VROWS;
                uint8_t* vb = vbuf + warp * Gm::VB_BYTES;
                const int prow = lane / WPP, qd = lane % WPP;
                const int cw = warp * Gm::CPW + 8 * qd;
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int f = 0; f < NF; ++f) {
                    const uint8_t* rowp = vr + (16 * kk + VROWS * f + prow) * CLD + 96 * (cw >> 7);
                    const uint32_t wq = *reinterpret_cast<const uint32_t*>(rowp + ((cw & 127) >> 1));
                    const uint32_t u = hi2_spread(*reinterpret_cast<const uint16_t*>(rowp + 64 + ((cw & 127) >> 2)));
                    *reinterpret_cast<uint4*>(vb + prow * VRS + 16 * qd) =
                        make_uint4(hi2_at<0>(nib64(wq, 0), u), hi2_at<1>(nib64(wq, 1), u), hi2_at<2>(nib64(wq, 2), u),
                                   hi2_at<3>(nib64(wq, 3), u));
                    __syncwarp();
                    uint32_t r0, r1, r2, r3;
                    if (VROWS == 8) {   // 8 positions, chunks 0..3 of 8 channels: m-tile chunk pairs
                        ldsm_x4_t(su32(vb + rr * VRS + 16 * mi), r0, r1, r2, r3);
                        ar[0][2 * f] = r0; ar[0][2 * f + 1] = r1;
                        ar[MT - 1][2 * f] = r2; ar[MT - 1][2 * f + 1] = r3;
                    } else {            // 16 positions, 16 channels: the four 8 x 8 tiles of one m-tile
                        ldsm_x4_t(su32(vb + (8 * (mi >> 1) + rr) * VRS + 16 * (mi & 1)), r0, r1, r2, r3);
                        ar[0][0] = r0; ar[0][1] = r1; ar[0][2] = r2; ar[0][3] = r3;
                    }
                    __syncwarp();
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int c0 = warp * (D / 8) + 16 * mt;
                uint32_t a0, a1, a2, a3;
                if (ring) {
                    a0 = ar[mt][0]; a1 = ar[mt][1]; a2 = ar[mt][2]; a3 = ar[mt][3];
                } else {
                    const int mi = lane >> 3, rr = lane & 7;
                    const int pos = 16 * kk + 8 * (mi >> 1) + rr, ch = c0 + 8 * (mi & 1);
                    ldsm_x4_t(su32(vr + pos * FLD + 2 * ch), a0, a1, a2, a3);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (bf) {
                        const uint2 bl = pb2[((8 + kk) * NT + nt) * 32 + lane];
                        mma_bf16(acc[mt][kk % C3][nt], a0, a1, a2, a3, bp[nt].x, bp[nt].y);
                        mma_bf16(acc[mt][kk % C3][nt], a0, a1, a2, a3, bl.x, bl.y);
                    } else {
                        mma16816(acc[mt][kk % C3][nt], a0, a1, a2, a3, bp[nt].x, bp[nt].y);
                    }
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) r[i] = acc[mt][0][nt][i] + (C3 == 2 ? acc[mt][C3 - 1][nt][i] : 0.f);
                const float z0 = ring ? 96.f * a1s[nt][0] : 0.f, z1 = ring ? 96.f * a1s[nt][1] : 0.f;
                O[mt][nt][0] = al[nt][0] * O[mt][nt][0] + (r[0] - z0);
                O[mt][nt][1] = al[nt][1] * O[mt][nt][1] + (r[1] - z1);
                O[mt][nt][2] = al[nt][0] * O[mt][nt][2] + (r[2] - z0);
                O[mt][nt][3] = al[nt][1] * O[mt][nt][3] + (r[3] - z1);
            }
        if (!ring) fence_async_smem();    // the zero fill above precedes the next bulk copy into this stage
    }

    // ---- partial: sums over rows and warps, o (ring: rotated back), m and l
    csync();
    if (threadIdx.x == 0 && s_abort) {   // a wait timed out: wait (bounded, fresh limit) for copies in flight
        s_abort = 0;
        mbar_wait(qbar, 0, status, &s_abort);
        for (int i = max(0, issued - nst); i < issued; ++i)
            mbar_wait(su32(&full[i % nst]), (i / nst) & 1, status, &s_abort);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float l = l_part[nt][c];
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (g == 0) red[(nt * 8 + 2 * tq + c) * 8 + warp] = l;
            if (warp == 0 && g == 0) red[2 * NQ * 8 + nt * 8 + 2 * tq + c] = m_run[nt][c];
        }
    csync();
    float* ofin = reinterpret_cast<float*>(stages);                     // [NQ][D], stages drained
    // channels of fragment rows g and g + 8: ring at D 256 (movmatrix tiles above) 8 (g >> 1) +
    // 2 mt + 4 (g & 1) of the warp's and the next one; ring at D 128 (ldmatrix of the staging
    // buffer) channels 0,4,1,5,2,6,3,7 of each 8-channel group; 16-bit rows in order
    const int cg = ring ? ((g >> 1) + 4 * (g & 1)) : g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int qc = nt * 8 + 2 * tq;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const bool mv = ring && Gm::CPW == 32;
            const int cA = mv ? warp * 32 + 8 * (g >> 1) + 2 * mt + 4 * (g & 1) : warp * (D / 8) + 16 * mt + cg;
            const int cB = mv ? cA + 1 : cA + 8;
            ofin[qc * D + cA] = O[mt][nt][0];
            ofin[(qc + 1) * D + cA] = O[mt][nt][1];
            ofin[qc * D + cB] = O[mt][nt][2];
            ofin[(qc + 1) * D + cB] = O[mt][nt][3];
        }
    }
    if (threadIdx.x < NQ) {
        const float4* r4 = reinterpret_cast<const float4*>(red + threadIdx.x * 8);
        const float4 x = r4[0], y = r4[1];
        red[2 * NQ * 8 + NQ + threadIdx.x] = ((x.x + x.y) + (x.z + x.w)) + ((y.x + y.y) + (y.z + y.w));
    }
    csync();
    if (p.early) grid_dep_wait();   // the merge ahead has read the partials buffer
    write_partial<D, NQ>(ofin, red + 2 * NQ * 8, red + 2 * NQ * 8 + NQ, p.partials + (size_t)item * (2 * NQ + NQ * D),
                         ring ? ROT : (int)ROT_NONE);
}

}  // namespace
}  // namespace kvq
