// Decode attention over sealed body records: the bandwidth-critical part of the path.
//
// One CTA of 8 warps per work item (sequence, KV head, run of 128-position groups), two CTAs
// per SM where shared memory allows. Thread 0 streams each group's K record and V record
// (contiguous, 16-byte multiples) into a ring of shared-memory stages with cp.async.bulk,
// completion tracked by mbarriers; a stage is refilled after the first barrier of the group
// that follows its last reader. All 8 warps consume each group:
//   0. (KVarN) the query fragments times the group's column scales, q' = q C in fp16, one
//      8-channel chunk per thread from the fp16 rotated query held in registers; barrier.
//   1. scores: warp w takes the 16 positions that value k-step w of step 3 covers and all D
//      channels, decoding K rows from shared memory straight into mma.sync m16n8k16 A
//      fragments (positions on M, the GQA query group on N); an mma with an all-ones A gives
//      sum_c q'_c per query for the offset / zero-point term. Epilogue: log2-domain scores,
//      the warp's maximum per query to shared memory; barrier; every thread forms the group
//      maximum, the rescale factor alpha, p = 2^(s - m) and its running sum (registers), and
//      P' = p x (value scale of the position) in fp16; movmatrix transposes the 16 x 8 P'
//      tile into the B-fragment order of step 3 (one 8-byte store per lane); barrier.
//   3. values: warp w takes channels [wD/8, (w+1)D/8) and all 128 positions, decoding V
//      rows (channel-major records: 16 bytes cover 32 positions of a channel) into A
//      fragments: O^T[ch][q] = alpha O^T + F (V^T P'^T + zero-point term).
// Codes enter the mma through the fp16 exponent trick: a 4-bit code n placed in mantissa bits
// 4-7 under exponent 6 reads exactly 64 + n (the fifth KVarN bit is mantissa bit 8, +16), a
// signed byte b reads 1152 + b. The offsets cancel against sum q' (scores) or sum P' (values):
// per group (values: an all-ones mma over the warp's P' copy gives sum P').
// The partial (m, l, o) is rotated back to the original domain and merged with the region
// partials by decode_merge_kernel (kernels_attn.cu).
#include "stream_common.cuh"
#include "region_item.cuh"

namespace kvq {
namespace {

// ------------------------------------------------------------------------------ geometry
// The rotation of a layout follows from its key format: HAD256 for KVarN, TBQ128 for TBQ4 and
// tq5_0 keys, none for the block formats (an instance compiles only its own rotation).
template <int KF>
constexpr int kRotOf = (KF == KF_KVARN) ? (int)ROT_HAD256 : ((KF == KF_TBQ4 || KF == KF_TQ5) ? (int)ROT_TBQ128 : (int)ROT_NONE);

template <int D, int NQ, int KF, int VF, int KB, int VB>
struct Geo {
    static constexpr int NT = NQ / 8;
    static constexpr int KS = D / 16;                                   // score k-steps
    // K fragment block: the channels one set of score accumulators covers. Q8_0 K is dequantised
    // in registers (code x block scale), so one block spans all D channels and each thread quad
    // owns a contiguous quarter of the row
    static constexpr int WK = (KF == KF_KVARN) ? 256 : ((KF == KF_TBQ4 || KF == KF_TQ5) ? 128 :
                                                       ((KF == KF_Q8 || KF == KF_Q51) ? D : 32));
    static constexpr int NBK = D / WK;
    static constexpr int KSPB = WK / 16;                                // k-steps per K block
    static constexpr int WV = (VF == KF_KVARN) ? 256 : (VF == KF_TBQ4 ? 128 : 32);   // V scale block
    static constexpr int NVB = D / WV;                                  // P' copies
    static constexpr int MT = D / 128;                                  // value m-tiles per warp
    static constexpr bool KNIB = (KF == KF_KVARN || KF == KF_Q4 || KF == KF_Q51 || KF == KF_TQ5);   // K pairs (x, x+4)
    static constexpr bool VNIB = (VF == KF_KVARN || VF == KF_Q4);
    // value the raw fp16 operand reads for code 0 (the code's own centre included)
    // Q5_1 keys are dequantised in the fragments (code x d + m); tq5_0 keys read 64 + code, the
    // code's centre 16 included
    static constexpr float KOFF = (KF == KF_KVARN) ? 64.f : (KF == KF_Q4 ? 72.f : (KF == KF_TQ5 ? 80.f : 0.f));
    static constexpr float VOFF = (VF == KF_KVARN) ? 64.f : (VF == KF_Q4 ? 72.f : (VF == KF_Q8 ? 1152.f : 0.f));
    static constexpr bool ZV = (VF == KF_KVARN);                        // per-group value zero-point sums
    static constexpr bool PSV = (VF == KF_Q8 || VF == KF_Q4);           // sum of P' per group (offset)
    static constexpr bool LUT = (KF == KF_TBQ4) || (VF == KF_TBQ4);
    static constexpr int rec(int f, int b) {
        return f == KF_KVARN ? (D / 256) * (4096 * b + 1152)
                             : (f == KF_TBQ4 ? 66 * D : (f == KF_Q8 ? 136 * D : (f == KF_Q51 ? 96 * D :
                                                                                 (f == KF_TQ5 ? 82 * D : 72 * D))));
    }
    static constexpr int REC_K = rec(KF, KB), REC_V = rec(VF, VB);
    static constexpr int V_OFF = (REC_K + 127) & ~127;
    static constexpr int STAGE = (V_OFF + REC_V + 127) & ~127;
    static constexpr int QB_BYTES = NT * KS * 256;                      // query fragments (= NQ D fp16)
    static constexpr int P_BYTES = NVB * 8 * NT * 256;                  // P' fragments
    static_assert(P_BYTES >= 2 * D, "the P' area stages the codes of a fused append");
    static constexpr int RED_FLOATS = (NVB + 2) * NQ * 8 + NQ;          // [q][warp] exchange rows, m, l
    // KVarN codes of 2 or 3 bits: each group's code planes are expanded in shared memory into
    // the 4-bit nibble image of a KVarN4 tile (16 KB per 256-channel tile), which the 4-bit
    // fragment decoders read; the scales are read from the staged record
    static constexpr bool KIMG = (KF == KF_KVARN) && (KB < 4);
    static constexpr bool VIMG = (VF == KF_KVARN) && (VB < 4);
    static constexpr int IMG_BYTES = ((KIMG ? 1 : 0) + (VIMG ? 1 : 0)) * 16384 * (D / 256);
    static constexpr int FIXED = 128 + (LUT ? kLutBytes : 0) + QB_BYTES + P_BYTES + RED_FLOATS * 4 + IMG_BYTES;
    // resident CTAs per SM: three when two stages fit in a third of shared memory, else two,
    // else one (the per-CTA budgets leave the 1 KB per CTA the SM reserves)
    static constexpr int THREE_CTA_BYTES = 74 * 1024;
    static constexpr int TWO_CTA_BYTES = 112 * 1024;
    static constexpr bool THREE = FIXED + 2 * STAGE <= THREE_CTA_BYTES;
    static constexpr bool TWO = FIXED + 2 * STAGE <= TWO_CTA_BYTES;
    static constexpr int MINB = THREE ? 3 : (TWO ? 2 : 1);
    static constexpr int BUDGET = THREE ? THREE_CTA_BYTES : (TWO ? TWO_CTA_BYTES : 227 * 1024);
    static constexpr int NTASK = NQ * D / 8;                            // 8-channel query chunks
    static constexpr int TPT = (NTASK + kCT - 1) / kCT;                 // chunks per consumer thread
};

// The N fp16 values of one position's scale row (16-byte aligned rows of N values), as floats.
template <int N>
__device__ __forceinline__ void load_row_f(const uint16_t* row, float (&f)[N]) {
    if constexpr (N == 1) {
        f[0] = h2f(row[0]);
    } else if constexpr (N == 2) {
        const float2 v = __half22float2(as_h2(*reinterpret_cast<const uint32_t*>(row)));
        f[0] = v.x; f[1] = v.y;
    } else if constexpr (N == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(row);
        const float2 a = __half22float2(as_h2(u.x)), b = __half22float2(as_h2(u.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
#pragma unroll
        for (int k = 0; k < N / 8; ++k) {
            const uint4 u = reinterpret_cast<const uint4*>(row)[k];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a = __half22float2(as_h2(w[i]));
                f[8 * k + 2 * i] = a.x;
                f[8 * k + 2 * i + 1] = a.y;
            }
        }
    }
}

// The centroid pair of byte k (0..3) of y from the lane-replicated table (entry e of lane l at
// byte offset 128 e + 4 l of lutb): a byte permute extracts e and one multiply-add forms the
// offset with lw = 4 l, so the integer pipe, which issues at half rate, takes one instruction
// per lookup and the multiply-add pipe the other.
template <int K>
__device__ __forceinline__ uint32_t lut_pair(const uint8_t* lutb, uint32_t y, uint32_t lw) {
    const uint32_t e = __byte_perm(y, 0u, 0x4440 | K);
    return *reinterpret_cast<const uint32_t*>(lutb + (e * 128u + lw));
}

// 8 codes of a 2-bit plane (16 bits, code m at bits 2m) spread to bits 4m, 4m + 1.
__device__ __forceinline__ uint32_t spread2(uint32_t x) {
    x = (x | (x << 8)) & 0x00FF00FFu;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    return (x | (x << 2)) & 0x33333333u;
}
// 8 codes of a 1-bit plane (a byte, code m at bit m) spread to bit 4m.
__device__ __forceinline__ uint32_t spread1(uint32_t x) {
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    return (x | (x << 3)) & 0x11111111u;
}
// The nibble image (KVarN4 layout) of the codes of ntile 2- or 3-bit KVarN tiles at rec: word u
// of a tile's image holds the 8 codes whose low bits are uint16 u of the 2-bit plane and whose
// third bits are byte u of the 1-bit plane; this is so for the token rows of K and the channel
// rows of V alike (the planes are row-major with the same codes per row). All threads.
template <int B>
__device__ __forceinline__ void nibble_image(const uint8_t* rec, int ntile, uint8_t* img) {
    for (int u = threadIdx.x; u < 4096 * ntile; u += kCT) {
        const uint8_t* tb = rec + (size_t)(u >> 12) * (4096 * B + 1152);
        const int uu = u & 4095;
        uint32_t x = spread2(reinterpret_cast<const uint16_t*>(tb)[uu]);
        if (B == 3) x |= spread1(tb[8192 + uu]) << 2;
        reinterpret_cast<uint32_t*>(img + (size_t)(u >> 12) * 16384)[uu] = x;
    }
}

// ------------------------------------------------------------------------------ a body item
// One body work item (partial index `item`: body items follow the region items), run by a CTA
// of 8 warps on the dynamic shared memory `smem` with nst stages; s_abort is the CTA's abort flag.
template <int D, int NQ, int KF, int VF, int KB, int VB>
__device__ __forceinline__ void body_item(const Layout& L, const AttnParams& p, const int item, const int nst,
                                          uint8_t* smem, int& s_abort) {
    using Gm = Geo<D, NQ, KF, VF, KB, VB>;
    constexpr int NT = Gm::NT, KS = Gm::KS, NBK = Gm::NBK, KSPB = Gm::KSPB, WK = Gm::WK;
    constexpr int NVB = Gm::NVB, WV = Gm::WV, MT = Gm::MT, TPT = Gm::TPT;

    int b = 0;
    while (b + 1 < p.n_seq && p.seq[b + 1].body_first <= item) ++b;
    const SeqSpan& sp = p.seq[b];
    const int local = item - sp.body_first;
    const int h = local / sp.body_per_head;
    const int kb_ = local % sp.body_per_head;             // the head's groups split evenly over its items
    // the head's groups split evenly: 32-bit products while they fit (items per head < 2^16)
    int g0, ngroups;
    if (sp.body_groups < (1 << 15)) {
        g0 = (kb_ * sp.body_groups) / sp.body_per_head;
        ngroups = ((kb_ + 1) * sp.body_groups) / sp.body_per_head - g0;
    } else {
        g0 = (int)((int64_t)kb_ * sp.body_groups / sp.body_per_head);
        ngroups = (int)((int64_t)(kb_ + 1) * sp.body_groups / sp.body_per_head) - g0;
    }
    const int64_t unit = L.unit(p.layer, sp.slot, h);
    uint32_t* status = status_word(L, p.pool);

    constexpr uint32_t recK = Gm::REC_K, recV = Gm::REC_V;
    constexpr uint32_t v_off = Gm::V_OFF, stage_bytes = Gm::STAGE;
    // the centroid-pair table first, at a fixed offset (its lookups then need no base address
    // arithmetic), the record stages after it
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem);
    uint8_t* stages = smem + (Gm::LUT ? kLutBytes : 0);
    uint8_t* tailp = stages + (size_t)nst * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(tailp);
    uint8_t* cur = tailp + 128;
    uint32_t* qb = reinterpret_cast<uint32_t*>(cur);      cur += Gm::QB_BYTES;
    uint32_t* pbuf = reinterpret_cast<uint32_t*>(cur);    cur += Gm::P_BYTES;
    float* red = reinterpret_cast<float*>(cur);
    float* zsm = red + NQ * 8;                            // [NVB][NQ][warp] value zero-point sums
    uint8_t* kimg = reinterpret_cast<uint8_t*>(red + Gm::RED_FLOATS);   // nibble images (2/3-bit codes)
    uint8_t* vimg = kimg + (Gm::KIMG ? 16384 * (D / 256) : 0);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // thread 0 streams the records: group i into stage i % nst, issued once stage i % nst is
    // free (the first barrier of group i - nst + 1 follows every read of group i - nst)
    const uint8_t* kb = body_rec(L, p.pool, 0, unit, g0);
    const uint8_t* vb = body_rec(L, p.pool, 1, unit, g0);
    int isl = 0;                                          // stage of the next issue (thread 0): issued % nst
    auto issue = [&](int i) {
        const int sl = isl;
        isl = (isl + 1 == nst) ? 0 : isl + 1;
        const uint32_t dst = su32(stages + (size_t)sl * stage_bytes);
        const uint32_t fb = su32(&full[sl]);
        mbar_expect_tx(fb, recK + recV);
        bulk_g2s(dst, kb + (size_t)i * recK, recK, fb);
        bulk_g2s(dst + v_off, vb + (size_t)i * recV, recV, fb);
    };
    // the query rows of the head (G x D fp16, contiguous) land in the fragment area first: the
    // set-up waits on them (full[4]) while the first groups' records stream in behind them
    const int G = L.G;
    const uint16_t* qsrc = p.q + ((int64_t)b * L.Hq + (int64_t)h * G) * D;
    const uint32_t qbar = su32(&full[4]);
    int issued = 0;
    const int g = lane >> 2, tq = lane & 3;
    // set-up that touches no global memory (the item from the launch parameters, the barriers,
    // the centroid-pair table from constant memory) runs before the wait for the launch ahead:
    // with programmatic serialization the CTA is placed while that launch drains
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < nst; ++i) mbar_init(su32(&full[i]), 1);
        mbar_init(qbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (Gm::LUT) {
        for (int i = threadIdx.x; i < 256 * 32; i += kCT) {
            const int by = i >> 5;
            lut[i] = pack_f2(c_tab.cent[by & 15], c_tab.cent[by >> 4]);
        }
    }
    if (!p.early) grid_dep_wait();
    if (threadIdx.x == 0) {
        mbar_expect_tx(qbar, (uint32_t)(G * D * 2));
        bulk_g2s(su32(qb), qsrc, (uint32_t)(G * D * 2), qbar);
        for (; issued < min(nst, ngroups); ++issued) issue(issued);
    }
    __syncthreads();
    if (p.knew != nullptr && kb_ == 0) {
        // fused decode step: the head's first body item appends the newest position (threads
        // 0-127 the K row, 128-255 the V row; codes staged in the P' area, unused yet) while its
        // first records are in flight. No item of this launch reads the slots written (the region
        // item that holds the newest position reads its row from the input).
        const int w = threadIdx.x >> 7;
        append_newest(L, p.pool, unit, w, sp.n_tok - 1, (w ? p.vnew : p.knew) + ((int64_t)b * L.H + h) * D,
                      threadIdx.x & 127, reinterpret_cast<uint8_t*>(pbuf) + w * D);
    }

    // ================================================================== consumers: set-up
    const uint8_t* lutb = reinterpret_cast<const uint8_t*>(lut);
    const uint32_t lw = (uint32_t)lane * 4u;
    __half* qr = reinterpret_cast<__half*>(qb);           // query rows, fp16 [NQ][D], rotated in place
    mbar_wait(qbar, 0, status, &s_abort);
    {
        const uint16_t* q = reinterpret_cast<const uint16_t*>(qr);
        constexpr int rot = kRotOf<KF>;
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

    // This thread's query chunks (8 consecutive channels of one query) in the order of the two
    // fragment entries they feed (k-steps j0, j0 + 1): KNIB pairs (0,4) (1,5) | (2,6) (3,7),
    // otherwise (0,1) (2,3) | (4,5) (6,7).
    uint32_t qv[TPT][4];
    int qe[TPT], qcoff[TPT];
#pragma unroll
    for (int k = 0; k < TPT; ++k) {
        const int t = threadIdx.x + kCT * k;
        qe[k] = -1;
        qcoff[k] = 0;
        qv[k][0] = qv[k][1] = qv[k][2] = qv[k][3] = 0u;
        if (t < Gm::NTASK) {
            // lanes of a warp take the 32 entries (query, quad) of one k-step pair: the stores
            // below are consecutive 8-byte words
            const int ln = t & 31, rest = t >> 5;
            const int tq_ = ln & 3, nt_ = rest % NT, jb = rest / NT;
            const int qi = nt_ * 8 + (ln >> 2);
            const int bb = jb / (WK / 32), m = jb % (WK / 32);
            const int ub = tq_ * (WK / 32) + m, u = bb * (WK / 8) + ub;
            const int j0 = bb * KSPB + 2 * m;
            qe[k] = (((qi >> 3) * KS + j0) * 8 + (qi & 7)) * 4 + tq_;
            qcoff[k] = bb * (4096 * KB + 1152) + 4096 * KB + 512 + 16 * ub;   // KVarN column scales
            const uint4 x = *reinterpret_cast<const uint4*>(qr + qi * D + 8 * u);
            if (Gm::KNIB) {
                qv[k][0] = __byte_perm(x.x, x.z, 0x5410);
                qv[k][1] = __byte_perm(x.x, x.z, 0x7632);
                qv[k][2] = __byte_perm(x.y, x.w, 0x5410);
                qv[k][3] = __byte_perm(x.y, x.w, 0x7632);
            } else {
                qv[k][0] = x.x; qv[k][1] = x.y; qv[k][2] = x.z; qv[k][3] = x.w;
            }
        }
    }
    csync();   // every chunk is read before the fragment area is rewritten
    // query fragments; KVarN: times the column scales of the group whose K record is at kr
    auto write_qb = [&](const uint8_t* kr) {
#pragma unroll
        for (int k = 0; k < TPT; ++k) {
            if (qe[k] < 0) continue;
            uint32_t v0 = qv[k][0], v1 = qv[k][1], v2 = qv[k][2], v3 = qv[k][3];
            if (KF == KF_KVARN) {
                const uint4 c = *reinterpret_cast<const uint4*>(kr + qcoff[k]);
                v0 = hmul2u(v0, __byte_perm(c.x, c.z, 0x5410));
                v1 = hmul2u(v1, __byte_perm(c.x, c.z, 0x7632));
                v2 = hmul2u(v2, __byte_perm(c.y, c.w, 0x5410));
                v3 = hmul2u(v3, __byte_perm(c.y, c.w, 0x7632));
            }
            uint2* e = reinterpret_cast<uint2*>(qb) + qe[k];
            e[0] = make_uint2(v0, v1);
            e[32] = make_uint2(v2, v3);
        }
    };
    const uint2* qb2 = reinterpret_cast<const uint2*>(qb);
    const uint2* pb2 = reinterpret_cast<const uint2*>(pbuf);
    constexpr uint32_t ONE2 = 0x3C003C00u;
    // sum of q' per K block for this thread's queries (columns 2tq, 2tq+1 of each n-tile)
    float zk[NBK][NT][2];
#pragma unroll
    for (int bk = 0; bk < NBK; ++bk)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) zk[bk][nt][0] = zk[bk][nt][1] = 0.f;
    // formats whose fragments are fixed per item keep them in registers (one n-tile)
    constexpr bool QREG = (KF != KF_KVARN) && (NT == 1);
    uint2 qf[QREG ? KS : 1];
    if (KF != KF_KVARN) {
        write_qb(nullptr);
        csync();
        if constexpr (QREG) {
#pragma unroll
            for (int j = 0; j < KS; ++j) qf[j] = qb2[(j * 8 + g) * 4 + tq];
        }
        if (Gm::KOFF != 0.f) {
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const uint2 bq = qb2[((nt * KS + bk * KSPB + jj) * 8 + g) * 4 + tq];
                        mma16816(a1, ONE2, ONE2, ONE2, ONE2, bq.x, bq.y);
                    }
                    zk[bk][nt][0] = a1[0];
                    zk[bk][nt][1] = a1[1];
                }
        }
    }

    // score rows g and g+8 of this warp: the positions value k-step `warp` feeds (see step 3)
    const int t0 = Gm::VNIB ? 32 * (g >> 1) + 8 * (warp >> 1) + 2 * (warp & 1) + 4 * (g & 1)
                            : 32 * (g >> 1) + 4 * warp + (g & 1);
    const int t1 = t0 + (Gm::VNIB ? 1 : 2);
    const int vw = (warp * (D / 8)) / WV;                 // value scale block of this warp's channels
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

    // the stage of group gi (gi % nst) and its barrier phase ((gi / nst) & 1), stepped per group
    int sl = 0;
    uint32_t phase = 0;
    for (int gi = 0; gi < ngroups; ++gi, sl = (sl + 1 == nst) ? 0 : sl + 1, phase ^= (sl == 0)) {
        mbar_wait(su32(&full[sl]), phase, status, &s_abort);
        const uint8_t* kr = stages + (size_t)sl * stage_bytes;
        const uint8_t* vr = kr + v_off;
        if constexpr (Gm::KIMG || Gm::VIMG) {
            csync();   // the previous group's reads of the images are done
            if constexpr (Gm::KIMG) nibble_image<KB>(kr, D / 256, kimg);
            if constexpr (Gm::VIMG) nibble_image<VB>(vr, D / 256, vimg);
        }
        if (KF == KF_KVARN) {
            write_qb(kr);
            csync();
            if (threadIdx.x == 0 && gi >= 1 && issued < ngroups) issue(issued++);
        }

        // ---------------- step 1: scores of positions t0, t1 (rows g, g+8), all channels
        float s4[NT][4];
        {
            // two accumulation chains per (block, n-tile), by k-step parity, so consecutive mma
            // do not wait on each other
            float acc[NBK][NT][2][4];
            float a1[NBK][NT][2][4];
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[bk][nt][0][i] = acc[bk][nt][1][i] = a1[bk][nt][0][i] = a1[bk][nt][1][i] = 0.f;
            // TBQ4: blocks of 128 channels, 16 bytes of this row and block per thread; with two
            // blocks, odd rows read them in the other order so a quarter warp hits 32 banks
            uint4 tY0[NBK], tY1[NBK];
            if (KF == KF_TBQ4 || KF == KF_TQ5) {
                const bool sw = (NBK == 2) && (g & 1);
#pragma unroll
                for (int bk = 0; bk < NBK; ++bk) {
                    const int bka = sw ? (NBK - 1 - bk) : bk;
                    tY0[bk] = *reinterpret_cast<const uint4*>(kr + t0 * (D / 2) + 64 * bka + 16 * tq);
                    tY1[bk] = *reinterpret_cast<const uint4*>(kr + t1 * (D / 2) + 64 * bka + 16 * tq);
                }
                if (NBK == 2 && sw) {
                    const uint4 a = tY0[0]; tY0[0] = tY0[NBK - 1]; tY0[NBK - 1] = a;
                    const uint4 c = tY1[0]; tY1[0] = tY1[NBK - 1]; tY1[NBK - 1] = c;
                }
            }
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk) {
                if (KF == KF_KVARN) {
                    // this thread's 64 channels of the 256-channel tile bk: 32 bytes per row; odd
                    // rows read the two halves in the other order so a quarter warp hits 32 banks
                    const uint8_t* tb = kr + (size_t)bk * (4096 * KB + 1152);
                    const uint8_t* tc = Gm::KIMG ? kimg + (size_t)bk * 16384 : tb;     // nibble codes
                    const int odd = g & 1;
                    uint4 x0a = *reinterpret_cast<const uint4*>(tc + t0 * 128 + 32 * tq + 16 * odd);
                    uint4 x0b = *reinterpret_cast<const uint4*>(tc + t0 * 128 + 32 * tq + 16 * (1 - odd));
                    uint4 x1a = *reinterpret_cast<const uint4*>(tc + t1 * 128 + 32 * tq + 16 * odd);
                    uint4 x1b = *reinterpret_cast<const uint4*>(tc + t1 * 128 + 32 * tq + 16 * (1 - odd));
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
                        const int m = jj >> 1, x = 2 * (jj & 1);
                        uint32_t a0 = nib64(W0[m], x), a2 = nib64(W0[m], x + 1);
                        uint32_t a1r = nib64(W1[m], x), a3 = nib64(W1[m], x + 1);
                        if (KB == 5) {
                            const int bx = 8 * (m & 3) + x;
                            const uint32_t h0 = (m < 4) ? H0.x : H0.y, h1 = (m < 4) ? H1.x : H1.y;
                            a0 = add_bit5(a0, h0, bx); a2 = add_bit5(a2, h0, bx + 1);
                            a1r = add_bit5(a1r, h1, bx); a3 = add_bit5(a3, h1, bx + 1);
                        }
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = QREG ? qf[QREG ? j : 0] : qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt][jj & 1], a0, a1r, a2, a3, bq.x, bq.y);
                            mma16816(a1[bk][nt][jj & 1], ONE2, ONE2, ONE2, ONE2, bq.x, bq.y);
                        }
                    }
                } else if (KF == KF_TBQ4) {
                    const uint4 y0 = tY0[bk], y1 = tY1[bk];
                    const uint32_t Y0[4] = {y0.x, y0.y, y0.z, y0.w}, Y1[4] = {y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int m = jj >> 1;
                        uint32_t a0, a2, a1r, a3;
                        if (jj & 1) {
                            a0 = lut_pair<2>(lutb, Y0[m], lw); a2 = lut_pair<3>(lutb, Y0[m], lw);
                            a1r = lut_pair<2>(lutb, Y1[m], lw); a3 = lut_pair<3>(lutb, Y1[m], lw);
                        } else {
                            a0 = lut_pair<0>(lutb, Y0[m], lw); a2 = lut_pair<1>(lutb, Y0[m], lw);
                            a1r = lut_pair<0>(lutb, Y1[m], lw); a3 = lut_pair<1>(lutb, Y1[m], lw);
                        }
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = QREG ? qf[QREG ? j : 0] : qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt][jj & 1], a0, a1r, a2, a3, bq.x, bq.y);
                        }
                    }
                } else if (KF == KF_Q8) {
                    // channels [tq D/4, (tq+1) D/4) of rows t0, t1 (k-step j: 4 bytes at 4j), in 16-byte
                    // loads, odd rows taking each pair of loads in the other order (banks); each code
                    // byte b becomes (1152 + b) - 1152 = b, times its 32-channel block scale
                    constexpr int CPT = D / 4, NL = CPT / 16, NSB = CPT / 32;
                    const int odd = g & 1;
                    uint32_t W0[CPT / 4], W1[CPT / 4];
#pragma unroll
                    for (int i = 0; i < NL; i += 2) {
                        uint4 y0a = *reinterpret_cast<const uint4*>(kr + t0 * D + CPT * tq + 16 * (i + odd));
                        uint4 y0b = *reinterpret_cast<const uint4*>(kr + t0 * D + CPT * tq + 16 * (i + 1 - odd));
                        uint4 y1a = *reinterpret_cast<const uint4*>(kr + t1 * D + CPT * tq + 16 * (i + odd));
                        uint4 y1b = *reinterpret_cast<const uint4*>(kr + t1 * D + CPT * tq + 16 * (i + 1 - odd));
                        if (odd) {
                            const uint4 t = y0a; y0a = y0b; y0b = t;
                            const uint4 u = y1a; y1a = y1b; y1b = u;
                        }
                        W0[4 * i] = y0a.x; W0[4 * i + 1] = y0a.y; W0[4 * i + 2] = y0a.z; W0[4 * i + 3] = y0a.w;
                        W0[4 * i + 4] = y0b.x; W0[4 * i + 5] = y0b.y; W0[4 * i + 6] = y0b.z; W0[4 * i + 7] = y0b.w;
                        W1[4 * i] = y1a.x; W1[4 * i + 1] = y1a.y; W1[4 * i + 2] = y1a.z; W1[4 * i + 3] = y1a.w;
                        W1[4 * i + 4] = y1b.x; W1[4 * i + 5] = y1b.y; W1[4 * i + 6] = y1b.z; W1[4 * i + 7] = y1b.w;
                    }
                    const uint16_t* dr = reinterpret_cast<const uint16_t*>(kr + 128 * D);
                    uint32_t s0[NSB], s1[NSB];
#pragma unroll
                    for (int b2 = 0; b2 < NSB; ++b2) {
                        const uint32_t h0 = dr[t0 * (D / 32) + NSB * tq + b2], h1 = dr[t1 * (D / 32) + NSB * tq + b2];
                        s0[b2] = h0 | (h0 << 16);
                        s1[b2] = h1 | (h1 << 16);
                    }
                    const __half2 c1152 = __float2half2_rn(1152.f);
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int b2 = jj / 8;
                        const uint32_t a0 = hmul2u(as_u(__hsub2(as_h2(i8raw(W0[jj], 0x5140)), c1152)), s0[b2]);
                        const uint32_t a2 = hmul2u(as_u(__hsub2(as_h2(i8raw(W0[jj], 0x7362)), c1152)), s0[b2]);
                        const uint32_t a1r = hmul2u(as_u(__hsub2(as_h2(i8raw(W1[jj], 0x5140)), c1152)), s1[b2]);
                        const uint32_t a3 = hmul2u(as_u(__hsub2(as_h2(i8raw(W1[jj], 0x7362)), c1152)), s1[b2]);
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = QREG ? qf[QREG ? j : 0] : qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt][jj & 1], a0, a1r, a2, a3, bq.x, bq.y);
                        }
                    }
                } else if (KF == KF_TQ5) {
                    // tq5_0: this thread's 32 channels of the 128-channel block (16 bytes of the
                    // nibble plane, preloaded) and their fifth bits (4 bytes of the one-bit plane,
                    // bit 8 m + e for channel 8 m + e): 64 + code, scale after the mma
                    const uint4 y0 = tY0[bk], y1 = tY1[bk];
                    const uint32_t Y0[4] = {y0.x, y0.y, y0.z, y0.w}, Y1[4] = {y1.x, y1.y, y1.z, y1.w};
                    const uint32_t H0 = *reinterpret_cast<const uint32_t*>(kr + 64 * D + t0 * (D / 8) + 16 * bk + 4 * tq);
                    const uint32_t H1 = *reinterpret_cast<const uint32_t*>(kr + 64 * D + t1 * (D / 8) + 16 * bk + 4 * tq);
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int m = jj >> 1, x = 2 * (jj & 1), bx = 8 * m + x;
                        const uint32_t a0 = add_bit5(nib64(Y0[m], x), H0, bx), a2 = add_bit5(nib64(Y0[m], x + 1), H0, bx + 1);
                        const uint32_t a1r = add_bit5(nib64(Y1[m], x), H1, bx), a3 = add_bit5(nib64(Y1[m], x + 1), H1, bx + 1);
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = QREG ? qf[QREG ? j : 0] : qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt][jj & 1], a0, a1r, a2, a3, bq.x, bq.y);
                        }
                    }
                } else if (KF == KF_Q51) {
                    // Q5_1 (D = 128): thread quad tq holds the 32-channel block tq (16 bytes of
                    // nibbles, 4 bytes of fifth bits per row) and dequantises in the fragments:
                    // (64 + code - 64) x d + m in fp16, one rounding. Odd rows load t1 before t0,
                    // so a quarter warp's two rows lie 64 bytes apart (all 32 banks).
                    static_assert(KF != KF_Q51 || D == 128, "Q5_1 keys: one 32-channel block per thread quad");
                    const int odd = g & 1;
                    const int ra = odd ? t1 : t0, rb = odd ? t0 : t1;
                    uint4 ya = *reinterpret_cast<const uint4*>(kr + ra * (D / 2) + 16 * tq);
                    uint4 yb = *reinterpret_cast<const uint4*>(kr + rb * (D / 2) + 16 * tq);
                    if (odd) { const uint4 t = ya; ya = yb; yb = t; }
                    const uint32_t Y0[4] = {ya.x, ya.y, ya.z, ya.w}, Y1[4] = {yb.x, yb.y, yb.z, yb.w};
                    const uint32_t H0 = *reinterpret_cast<const uint32_t*>(kr + 64 * D + t0 * (D / 8) + 4 * tq);
                    const uint32_t H1 = *reinterpret_cast<const uint32_t*>(kr + 64 * D + t1 * (D / 8) + 4 * tq);
                    const uint16_t* dr = reinterpret_cast<const uint16_t*>(kr + 80 * D);
                    const uint16_t* mr = reinterpret_cast<const uint16_t*>(kr + 88 * D);
                    const uint32_t d0 = dr[t0 * 4 + tq], d1 = dr[t1 * 4 + tq];
                    const uint32_t m0 = mr[t0 * 4 + tq], m1 = mr[t1 * 4 + tq];
                    const __half2 dd0 = as_h2(d0 | (d0 << 16)), dd1 = as_h2(d1 | (d1 << 16));
                    const __half2 mm0 = as_h2(m0 | (m0 << 16)), mm1 = as_h2(m1 | (m1 << 16));
                    const __half2 c64 = __float2half2_rn(64.f);
                    auto deq = [&](uint32_t raw, __half2 d, __half2 mz) {
                        return as_u(__hfma2(__hsub2(as_h2(raw), c64), d, mz));
                    };
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int m = jj >> 1, x = 2 * (jj & 1), bx = 8 * m + x;
                        const uint32_t a0 = deq(add_bit5(nib64(Y0[m], x), H0, bx), dd0, mm0);
                        const uint32_t a2 = deq(add_bit5(nib64(Y0[m], x + 1), H0, bx + 1), dd0, mm0);
                        const uint32_t a1r = deq(add_bit5(nib64(Y1[m], x), H1, bx), dd1, mm1);
                        const uint32_t a3 = deq(add_bit5(nib64(Y1[m], x + 1), H1, bx + 1), dd1, mm1);
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = QREG ? qf[QREG ? j : 0] : qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt][jj & 1], a0, a1r, a2, a3, bq.x, bq.y);
                        }
                    }
                } else {   // Q4_0 K: one word of 8 nibbles per row and block
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(kr + t0 * (D / 2) + 16 * bk + 4 * tq);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(kr + t1 * (D / 2) + 16 * bk + 4 * tq);
#pragma unroll
                    for (int jj = 0; jj < KSPB; ++jj) {
                        const int x = 2 * jj;
                        const uint32_t a0 = nib64(w0, x), a2 = nib64(w0, x + 1);
                        const uint32_t a1r = nib64(w1, x), a3 = nib64(w1, x + 1);
                        const int j = bk * KSPB + jj;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 bq = QREG ? qf[QREG ? j : 0] : qb2[((nt * KS + j) * 8 + g) * 4 + tq];
                            mma16816(acc[bk][nt][jj & 1], a0, a1r, a2, a3, bq.x, bq.y);
                        }
                    }
                }
            }
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[bk][nt][0][i] += acc[bk][nt][1][i];
                        a1[bk][nt][0][i] += a1[bk][nt][1][i];
                    }
            // s = sum over K blocks of e(t) (acc - off sum q') + z(t) sum q', log2 domain; the
            // per-position block scales of TBQ4 / Q8_0 / Q4_0 come in one vector load per row
            float ek0[NBK], ek1[NBK];
            if (KF != KF_KVARN && KF != KF_Q8 && KF != KF_Q51) {
                const uint16_t* er = reinterpret_cast<const uint16_t*>(
                    kr + (KF == KF_TBQ4 ? 64 : (KF == KF_TQ5 ? 80 : 64)) * D);
                load_row_f<NBK>(er + t0 * NBK, ek0);
                load_row_f<NBK>(er + t1 * NBK, ek1);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) s4[nt][0] = s4[nt][1] = s4[nt][2] = s4[nt][3] = 0.f;
#pragma unroll
            for (int bk = 0; bk < NBK; ++bk) {
                float e0, e1, z0 = 0.f, z1 = 0.f;
                if (KF == KF_KVARN) {
                    const uint16_t* sb =
                        reinterpret_cast<const uint16_t*>(kr + (size_t)bk * (4096 * KB + 1152) + 4096 * KB);
                    e0 = h2f(sb[t0]); e1 = h2f(sb[t1]);
                    z0 = h2f(sb[128 + t0]); z1 = h2f(sb[128 + t1]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        zk[bk][nt][0] = a1[bk][nt][0][0];
                        zk[bk][nt][1] = a1[bk][nt][0][1];
                    }
                } else if (KF == KF_Q8 || KF == KF_Q51) {
                    e0 = e1 = 1.f;                  // dequantised in the fragments
                } else {
                    e0 = ek0[bk];
                    e1 = ek1[bk];
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float y0 = zk[bk][nt][0], y1 = zk[bk][nt][1];
                    if (Gm::KOFF != 0.f) {
                        const float o0 = Gm::KOFF * y0, o1 = Gm::KOFF * y1;
                        s4[nt][0] += e0 * (acc[bk][nt][0][0] - o0) + z0 * y0;
                        s4[nt][1] += e0 * (acc[bk][nt][0][1] - o1) + z0 * y1;
                        s4[nt][2] += e1 * (acc[bk][nt][0][2] - o0) + z1 * y0;
                        s4[nt][3] += e1 * (acc[bk][nt][0][3] - o1) + z1 * y1;
                    } else {
                        s4[nt][0] += e0 * acc[bk][nt][0][0];
                        s4[nt][1] += e0 * acc[bk][nt][0][1];
                        s4[nt][2] += e1 * acc[bk][nt][0][2];
                        s4[nt][3] += e1 * acc[bk][nt][0][3];
                    }
                }
            }
        }
        // the warp's maximum per query
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float mx0, mx1;
#pragma unroll
            for (int i = 0; i < 4; ++i) s4[nt][i] *= sc;
            mx0 = fmaxf(s4[nt][0], s4[nt][2]);
            mx1 = fmaxf(s4[nt][1], s4[nt][3]);
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
        if (KF != KF_KVARN && threadIdx.x == 0 && gi >= 1 && issued < ngroups) issue(issued++);

        // ---------------- step 2: group maximum, p, running sums, P' fragments
        float al[NT][2];
        float pr[NT][4];
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
        float fv0[NVB], fv1[NVB];
        if (VF != KF_KVARN) {
            const uint16_t* fr = reinterpret_cast<const uint16_t*>(vr + (VF == KF_Q8 ? 128 : 64) * D);
            load_row_f<NVB>(fr + t0 * NVB, fv0);
            load_row_f<NVB>(fr + t1 * NVB, fv1);
        }
#pragma unroll
        for (int v = 0; v < NVB; ++v) {
            float f0, f1, z0 = 0.f, z1 = 0.f;
            if (VF == KF_KVARN) {
                const uint16_t* sb =
                    reinterpret_cast<const uint16_t*>(vr + (size_t)v * (4096 * VB + 1152) + 4096 * VB);
                f0 = h2f(sb[t0]); f1 = h2f(sb[t1]);
                z0 = h2f(sb[128 + t0]); z1 = h2f(sb[128 + t1]);
            } else {
                f0 = fv0[v];
                f1 = fv1[v];
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t P0 = pack_f2(pr[nt][0] * f0, pr[nt][1] * f0);   // position t0, queries 2tq, 2tq+1
                const uint32_t P1 = pack_f2(pr[nt][2] * f1, pr[nt][3] * f1);   // position t1
                if (Gm::ZV) {
                    float zc0 = pr[nt][0] * z0 + pr[nt][2] * z1 - Gm::VOFF * (lo_f(P0) + lo_f(P1));
                    float zc1 = pr[nt][1] * z0 + pr[nt][3] * z1 - Gm::VOFF * (hi_f(P0) + hi_f(P1));
#pragma unroll
                    for (int o = 4; o <= 16; o <<= 1) {
                        zc0 += __shfl_xor_sync(0xffffffffu, zc0, o);
                        zc1 += __shfl_xor_sync(0xffffffffu, zc1, o);
                    }
                    if (g == 0) {
                        zsm[(v * NQ + nt * 8 + 2 * tq) * 8 + warp] = zc0;
                        zsm[(v * NQ + nt * 8 + 2 * tq + 1) * 8 + warp] = zc1;
                    }
                }
                reinterpret_cast<uint2*>(pbuf)[((v * 8 + warp) * NT + nt) * 32 + lane] =
                    make_uint2(movtrans(P0), movtrans(P1));
            }
        }
        csync();

        // ---------------- step 3: O^T[ch][q] = alpha O^T + F (V^T P'^T + z) for this warp's channels
        float zv[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            zv[nt][0] = zv[nt][1] = 0.f;
            if (Gm::ZV) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float4* r4 = reinterpret_cast<const float4*>(zsm + (vw * NQ + nt * 8 + 2 * tq + c) * 8);
                    const float4 x = r4[0], y = r4[1];
                    zv[nt][c] = ((x.x + x.y) + (x.z + x.w)) + ((y.x + y.y) + (y.z + y.w));
                }
            }
        }
        // rows of every m-tile first, then k-steps outer / m-tiles inner: the m-tiles' mma chains
        // interleave (a single m-tile splits its chain by k-step parity)
        constexpr int C3 = (MT == 1) ? 2 : 1;
        float acc[MT][C3][NT][4];
        uint32_t X0[MT][8], X1[MT][8];
        uint32_t H0[MT], H1[MT];
        const uint8_t* vt[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int c0 = warp * (D / 8) + 16 * mt + g, c1 = c0 + 8;
#pragma unroll
            for (int ch = 0; ch < C3; ++ch)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[mt][ch][nt][0] = acc[mt][ch][nt][1] = acc[mt][ch][nt][2] = acc[mt][ch][nt][3] = 0.f;
            H0[mt] = H1[mt] = 0;
            vt[mt] = vr;
            if (VF == KF_KVARN) {
                vt[mt] = vr + (size_t)(c0 >> 8) * (4096 * VB + 1152);
                const uint8_t* vc = Gm::VIMG ? vimg + (size_t)(c0 >> 8) * 16384 : vt[mt];   // nibble codes
                const uint4 y0 = *reinterpret_cast<const uint4*>(vc + (c0 & 255) * 64 + 16 * tq);
                const uint4 y1 = *reinterpret_cast<const uint4*>(vc + (c1 & 255) * 64 + 16 * tq);
                X0[mt][0] = y0.x; X0[mt][1] = y0.y; X0[mt][2] = y0.z; X0[mt][3] = y0.w;
                X1[mt][0] = y1.x; X1[mt][1] = y1.y; X1[mt][2] = y1.z; X1[mt][3] = y1.w;
                if (VB == 5) {
                    H0[mt] = *reinterpret_cast<const uint32_t*>(vt[mt] + 16384 + (c0 & 255) * 16 + 4 * tq);
                    H1[mt] = *reinterpret_cast<const uint32_t*>(vt[mt] + 16384 + (c1 & 255) * 16 + 4 * tq);
                }
            } else if (VF == KF_TBQ4 || VF == KF_Q4) {
                const uint4 y0 = *reinterpret_cast<const uint4*>(vr + c0 * 64 + 16 * tq);
                const uint4 y1 = *reinterpret_cast<const uint4*>(vr + c1 * 64 + 16 * tq);
                X0[mt][0] = y0.x; X0[mt][1] = y0.y; X0[mt][2] = y0.z; X0[mt][3] = y0.w;
                X1[mt][0] = y1.x; X1[mt][1] = y1.y; X1[mt][2] = y1.z; X1[mt][3] = y1.w;
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
                X0[mt][0] = y0a.x; X0[mt][1] = y0a.y; X0[mt][2] = y0a.z; X0[mt][3] = y0a.w;
                X0[mt][4] = y0b.x; X0[mt][5] = y0b.y; X0[mt][6] = y0b.z; X0[mt][7] = y0b.w;
                X1[mt][0] = y1a.x; X1[mt][1] = y1a.y; X1[mt][2] = y1a.z; X1[mt][3] = y1a.w;
                X1[mt][4] = y1b.x; X1[mt][5] = y1b.y; X1[mt][6] = y1b.z; X1[mt][7] = y1b.w;
            }
        }
        // Q8_0 / Q4_0 values: an all-ones mma sums this warp's P' copy (the code offset term)
        float a1v[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) a1v[nt][0] = a1v[nt][1] = a1v[nt][2] = a1v[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint2 bp[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                bp[nt] = pb2[((vw * 8 + kk) * NT + nt) * 32 + lane];
                if (Gm::PSV) mma16816(a1v[nt], ONE2, ONE2, ONE2, ONE2, bp[nt].x, bp[nt].y);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a0, a1r, a2, a3;
                if (Gm::VNIB) {
                    const int m = kk >> 1, x = 2 * (kk & 1);
                    a0 = nib64(X0[mt][m], x); a2 = nib64(X0[mt][m], x + 1);
                    a1r = nib64(X1[mt][m], x); a3 = nib64(X1[mt][m], x + 1);
                    if (VF == KF_KVARN && VB == 5) {
                        const int bx = 8 * m + x;
                        a0 = add_bit5(a0, H0[mt], bx); a2 = add_bit5(a2, H0[mt], bx + 1);
                        a1r = add_bit5(a1r, H1[mt], bx); a3 = add_bit5(a3, H1[mt], bx + 1);
                    }
                } else if (VF == KF_TBQ4) {
                    const int m = kk >> 1;
                    if (kk & 1) {
                        a0 = lut_pair<2>(lutb, X0[mt][m], lw); a2 = lut_pair<3>(lutb, X0[mt][m], lw);
                        a1r = lut_pair<2>(lutb, X1[mt][m], lw); a3 = lut_pair<3>(lutb, X1[mt][m], lw);
                    } else {
                        a0 = lut_pair<0>(lutb, X0[mt][m], lw); a2 = lut_pair<1>(lutb, X0[mt][m], lw);
                        a1r = lut_pair<0>(lutb, X1[mt][m], lw); a3 = lut_pair<1>(lutb, X1[mt][m], lw);
                    }
                } else {
                    a0 = i8raw(X0[mt][kk], 0x5140); a2 = i8raw(X0[mt][kk], 0x7362);
                    a1r = i8raw(X1[mt][kk], 0x5140); a3 = i8raw(X1[mt][kk], 0x7362);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816(acc[mt][kk % C3][nt], a0, a1r, a2, a3, bp[nt].x, bp[nt].y);
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int c0 = warp * (D / 8) + 16 * mt + g, c1 = c0 + 8;
            if (C3 == 2) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[mt][0][nt][i] += acc[mt][C3 - 1][nt][i];
            }
            float F0 = 1.f, F1 = 1.f;
            if (VF == KF_KVARN) {
                const uint16_t* sb = reinterpret_cast<const uint16_t*>(vt[mt] + 4096 * VB);
                F0 = h2f(sb[256 + (c0 & 255)]);
                F1 = h2f(sb[256 + (c1 & 255)]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float u0 = Gm::PSV ? zv[nt][0] - Gm::VOFF * a1v[nt][0] : zv[nt][0];
                const float u1 = Gm::PSV ? zv[nt][1] - Gm::VOFF * a1v[nt][1] : zv[nt][1];
                O[mt][nt][0] = al[nt][0] * O[mt][nt][0] + F0 * (acc[mt][0][nt][0] + u0);
                O[mt][nt][1] = al[nt][1] * O[mt][nt][1] + F0 * (acc[mt][0][nt][1] + u1);
                O[mt][nt][2] = al[nt][0] * O[mt][nt][2] + F1 * (acc[mt][0][nt][2] + u0);
                O[mt][nt][3] = al[nt][1] * O[mt][nt][3] + F1 * (acc[mt][0][nt][3] + u1);
            }
        }
    }

    // ---- partial: running sums over rows and warps, o rotated back to the original domain
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
            if (warp == 0 && g == 0) red[(NVB + 1) * NQ * 8 + nt * 8 + 2 * tq + c] = m_run[nt][c];
        }
    csync();
    float* ofin = reinterpret_cast<float*>(stages);                     // [NQ][D], stages drained
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int qc = nt * 8 + 2 * tq;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int c0 = warp * (D / 8) + 16 * mt + g;
            ofin[qc * D + c0] = O[mt][nt][0];
            ofin[(qc + 1) * D + c0] = O[mt][nt][1];
            ofin[qc * D + c0 + 8] = O[mt][nt][2];
            ofin[(qc + 1) * D + c0 + 8] = O[mt][nt][3];
        }
    }
    if (threadIdx.x < NQ) {
        const float4* r4 = reinterpret_cast<const float4*>(red + threadIdx.x * 8);
        const float4 x = r4[0], y = r4[1];
        red[(NVB + 1) * NQ * 8 + NQ + threadIdx.x] = ((x.x + x.y) + (x.z + x.w)) + ((y.x + y.y) + (y.z + y.w));
    }
    csync();
    if (p.early) grid_dep_wait();   // the merge ahead has read the partials buffer
    write_partial<D, NQ>(ofin, red + (NVB + 1) * NQ * 8, red + (NVB + 1) * NQ * 8 + NQ,
                         p.partials + (size_t)item * (2 * NQ + NQ * D), kRotOf<KF>);
}

// ------------------------------------------------------------------------------ the kernel
// Decode attention over one call's work list: CTAs [0, n_body) take the body items (the long
// ones, so they start first), the rest the region items (tq6_0 ring, 16-bit rows).
template <int D, int NQ, int KF, int VF, int KB, int VB, int RK>
__global__ void __launch_bounds__(kCT, (Geo<D, NQ, KF, VF, KB, VB>::MINB))
decode_attn_kernel(const __grid_constant__ Layout L, const __grid_constant__ AttnParams p, int n_body, int nst) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort;
    // launched with programmatic serialization, the CTAs may be placed while the launch ahead
    // drains: each item waits for it (grid_dep_wait) before it reads or writes global memory,
    // or, after the previous layer's merge (p.early), before it writes its partial
    if (p.region_first) {
        if ((int)blockIdx.x < p.n_region_items)
            region_item<D, NQ, RK, kRotOf<KF>>(L, p, (int)blockIdx.x, smem, s_abort);
        else
            body_item<D, NQ, KF, VF, KB, VB>(L, p, (int)blockIdx.x, nst, smem, s_abort);
    } else if ((int)blockIdx.x < n_body) {
        body_item<D, NQ, KF, VF, KB, VB>(L, p, p.n_region_items + (int)blockIdx.x, nst, smem, s_abort);
    } else {
        region_item<D, NQ, RK, kRotOf<KF>>(L, p, (int)blockIdx.x - n_body, smem, s_abort);
    }
}

// ------------------------------------------------------------------------------ launch
template <int D, int NQ, int KF, int VF, int KB, int VB>
int nstages(const Layout& L) {
    using Gm = Geo<D, NQ, KF, VF, KB, VB>;
    if (L.rec_bytes[0] != Gm::REC_K || L.rec_bytes[1] != Gm::REC_V) return 0;
    const size_t stage = Gm::STAGE;
    const size_t budget = Gm::BUDGET;
    if ((size_t)Gm::FIXED >= budget) return 0;
    int nst = (int)((budget - Gm::FIXED) / stage);
    if (nst > 4) nst = 4;
    if ((size_t)nst * stage < (size_t)NQ * D * 4) return 0;      // the final rows reuse the stages
    return nst >= 2 ? nst : 0;
}

// The region kinds a layout can hold: bit 0 a tq6_0 ring, bit 1 bf16 rows (journal or tail).
inline int region_kinds(const Layout& L) {
    return (L.journal == KVQ_TQ6_0 ? 1 : 0) | ((L.journal == KVQ_BF16 || L.tail_fmt == KVQ_BF16) ? 2 : 0);
}

template <int D, int NQ, int KF, int VF, int KB, int VB, int RK>
int launch_t(const Layout& L, const AttnParams& p, int n_body, int n_region, cudaStream_t st, bool pdl) {
    using Gm = Geo<D, NQ, KF, VF, KB, VB>;
    const int nst = nstages<D, NQ, KF, VF, KB, VB>(L);
    if (nst == 0) return (int)cudaErrorInvalidConfiguration;
    size_t smem = (size_t)nst * Gm::STAGE + Gm::FIXED;
    if (n_region > 0) {
        const size_t sr = (size_t)RGeo<D, NQ>::smem(L.tail_fmt == KVQ_BF16 || L.journal == KVQ_BF16);
        smem = smem > sr ? smem : sr;
    }
    auto kern = decode_attn_kernel<D, NQ, KF, VF, KB, VB, RK>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    const cudaError_t e = launch_k(kern, dim3(n_body + n_region), dim3(kCT), smem, st, pdl, L, p, n_body, nst);
    return e != cudaSuccess ? (int)e : (int)cudaGetLastError();
}

// Instantiated combinations (head_dim, query tile, K format, V format); other layouts keep
// their body positions in the region kernel's generic path.
template <typename F>
int dispatch(const Layout& L, F&& f) {
    const int k = L.fmt[0], v = L.fmt[1];
    const int rk = region_kinds(L);
    // SPEC: the region kinds of the workloads' layout for that case, which gets an instance of
    // its own (only those region readers: less code); other layouts take the generic instance
#define KVQ_BODY_CASE(D_, NQ_, KF_, VF_, KB_, VB_, KFMT, VFMT, SPEC)                            \
    if (L.D == D_ && L.NQ == NQ_ && k == KFMT && v == VFMT) {                                    \
        if (SPEC != 3 && rk == SPEC) return f.template run<D_, NQ_, KF_, VF_, KB_, VB_, SPEC>(); \
        return f.template run<D_, NQ_, KF_, VF_, KB_, VB_, 3>();                                 \
    }
    KVQ_BODY_CASE(128, 8, KF_TBQ4, KF_TBQ4, 4, 4, KVQ_TBQ4, KVQ_TBQ4, 0)
    KVQ_BODY_CASE(256, 8, KF_TBQ4, KF_TBQ4, 4, 4, KVQ_TBQ4, KVQ_TBQ4, 1)
    KVQ_BODY_CASE(256, 16, KF_TBQ4, KF_TBQ4, 4, 4, KVQ_TBQ4, KVQ_TBQ4, 3)
    KVQ_BODY_CASE(128, 8, KF_Q8, KF_Q4, 4, 4, KVQ_Q8_0, KVQ_Q4_0, 2)
    KVQ_BODY_CASE(128, 16, KF_Q8, KF_Q4, 4, 4, KVQ_Q8_0, KVQ_Q4_0, 3)
    KVQ_BODY_CASE(256, 8, KF_KVARN, KF_KVARN, 4, 4, KVQ_KVARN4, KVQ_KVARN4, 1)
    KVQ_BODY_CASE(256, 16, KF_KVARN, KF_KVARN, 4, 4, KVQ_KVARN4, KVQ_KVARN4, 3)
    KVQ_BODY_CASE(256, 8, KF_KVARN, KF_KVARN, 3, 2, KVQ_KVARN3, KVQ_KVARN2, 1)
    KVQ_BODY_CASE(512, 8, KF_KVARN, KF_KVARN, 5, 5, KVQ_KVARN5, KVQ_KVARN5, 3)
    KVQ_BODY_CASE(512, 16, KF_KVARN, KF_KVARN, 5, 5, KVQ_KVARN5, KVQ_KVARN5, 0)
    KVQ_BODY_CASE(128, 8, KF_Q51, KF_Q4, 5, 4, KVQ_Q5_1, KVQ_Q4_0, 2)
    KVQ_BODY_CASE(256, 8, KF_TQ5, KF_TBQ4, 5, 4, KVQ_TQ5_0, KVQ_TBQ4, 1)
#undef KVQ_BODY_CASE
    return -1;
}

struct CtasFn {
    const Layout& L;
    bool regions;
    template <int D, int NQ, int KF, int VF, int KB, int VB, int RK>
    int run() {
        using Gm = Geo<D, NQ, KF, VF, KB, VB>;
        const int nst = nstages<D, NQ, KF, VF, KB, VB>(L);
        if (nst == 0) return 0;
        if (!regions) return Gm::MINB;
        // the SM's 228 KB less 1 KB per CTA, shared by CTAs of the larger of the two footprints
        size_t smem = (size_t)nst * Gm::STAGE + Gm::FIXED;
        const size_t sr = (size_t)RGeo<D, NQ>::smem(L.tail_fmt == KVQ_BF16 || L.journal == KVQ_BF16);
        smem = smem > sr ? smem : sr;
        const int by_smem = (int)((228 * 1024) / (smem + 1024));
        return by_smem < Gm::MINB ? by_smem : Gm::MINB;
    }
};
struct LaunchFn {
    const Layout& L;
    const AttnParams& p;
    int n_body, n_region;
    cudaStream_t s;
    bool pdl;
    template <int D, int NQ, int KF, int VF, int KB, int VB, int RK>
    int run() { return launch_t<D, NQ, KF, VF, KB, VB, RK>(L, p, n_body, n_region, s, pdl); }
};

// The bounded wait's timeout path, exercised on purpose (a test launch): one CTA, thread 0
// arms barrier a for a 256-byte bulk copy of the pool's status area and issues it, and arms
// barrier b for 16 bytes that no copy ever delivers. The wait on b runs out after limit_ns
// (bit 1 of the status word, the CTA's abort flag); the wait on a, with the flag cleared and a
// fresh limit, completes, so the CTA retires with no copy in flight.
__global__ void wait_probe_kernel(const __grid_constant__ Layout L, const void* pool, uint64_t limit_ns) {
    __shared__ __align__(128) uint8_t buf[256];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int s_abort;
    if (threadIdx.x != 0) return;
    uint32_t* status = status_word(L, pool);
    s_abort = 0;
    const uint32_t a = su32(&bars[0]), b = su32(&bars[1]);
    mbar_init(a, 1);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    mbar_expect_tx(a, 256);
    bulk_g2s(su32(buf), pool, 256, a);
    mbar_expect_tx(b, 16);
    mbar_wait_ns(b, 0, status, &s_abort, limit_ns);
    s_abort = 0;
    mbar_wait_ns(a, 0, status, &s_abort, kWaitNs);
}

}  // namespace

int launch_wait_probe(const Layout& L, const void* pool, uint64_t limit_ns, void* stream) {
    wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(L, pool, limit_ns);
    return (int)cudaGetLastError();
}

int upload_tables_body(const FormatTables& t) {
    return (int)cudaMemcpyToSymbol(c_tab, &t, sizeof(FormatTables));
}

// Resident decode-kernel CTAs per SM for this layout (1 to 3), 0 when no instance fits it.
int body_ctas_per_sm(const Layout& L) {
    CtasFn f{L, false};
    const int r = dispatch(L, f);
    return r > 0 ? r : 0;
}

// Resident CTAs per SM of the decode kernel when it also takes the region items.
int decode_ctas_per_sm(const Layout& L) {
    CtasFn f{L, true};
    const int r = dispatch(L, f);
    return r > 0 ? r : 0;
}

// 1 when the streaming kernel takes this layout's region items: head_dim 128 or 256 (the ring,
// when present, in runs of whole 128-slot chunks), or 512 with 16-bit rows only.
int region_kernel_ok(const Layout& L) {
    if (L.D != 128 && L.D != 256 && L.D != 512) return 0;
    if (L.D == 512 && L.journal == KVQ_TQ6_0) return 0;
    if (L.journal == KVQ_TQ6_0 && L.R % 128 != 0) return 0;
    return 1;
}

// Launches the decode kernel over the body items and the first n_region region items of p.
int launch_decode_fused(const Layout& L, const AttnParams& p, int n_body, int n_region, void* stream, bool pdl) {
    if (n_body + n_region <= 0) return 0;
    LaunchFn f{L, p, n_body, n_region, (cudaStream_t)stream, pdl};
    const int r = dispatch(L, f);
    return r < 0 ? (int)cudaErrorInvalidValue : r;
}

}  // namespace kvq
