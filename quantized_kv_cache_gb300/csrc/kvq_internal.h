// Internal definitions shared by the host library and the CUDA kernels of the rotated
// low-bit KV cache: the device-pool layout, per-format record geometry and the launch
// parameter blocks. Not part of the public C ABI (include/kvq.h).
#pragma once

#include <cstdint>
#include <cstddef>
#include "../../include/kvq.h"

struct kvq_cache;

#ifdef __CUDACC__
#define KVQ_HD __host__ __device__ __forceinline__
#else
#define KVQ_HD inline
#endif

namespace kvq {

constexpr int kSink = 128;      // SJ-KVaRN §2.1: first 128 positions kept at 16 bits
constexpr int kGroup = 128;     // SJ-KVaRN §2.1: 128-token groups
constexpr int kMaxSeqPerCall = 32;   // keeps every launch parameter block under 4 KB
constexpr int kMaxG = 16;       // query heads per KV head handled by the decode kernel

enum Rot : int32_t { ROT_NONE = 0, ROT_HAD256 = 1, ROT_TBQ128 = 2 };

// Code bits of a KVarN body format, 0 for any other format.
KVQ_HD int kvarn_bits(int fmt) {
    switch (fmt) {
        case KVQ_KVARN2: return 2;
        case KVQ_KVARN3: return 3;
        case KVQ_KVARN4: return 4;
        case KVQ_KVARN5: return 5;
        case KVQ_KVARN6: return 6;
        case KVQ_KVARN8: return 8;
        default: return 0;
    }
}

// Code planes of a b-bit KVarN code, low plane first: plane i holds bits [s, s + w_i) of every
// code, s the widths before it (2: 2; 3: 2+1; 4: 4; 5: 4+1; 6: 4+2; 8: 8). A plane of width w
// packs each row's codes LSB-first, code i at bit w (i mod 8/w) of byte (i w) / 8; it spans
// 4,096 w bytes of a 128 x 256 tile. Returns the plane count; w[] receives the widths.
KVQ_HD int kvarn_planes(int bits, int* w) {
    switch (bits) {
        case 2: w[0] = 2; return 1;
        case 3: w[0] = 2; w[1] = 1; return 2;
        case 4: w[0] = 4; return 1;
        case 5: w[0] = 4; w[1] = 1; return 2;
        case 6: w[0] = 4; w[1] = 2; return 2;
        case 8: w[0] = 8; return 1;
        default: return 0;
    }
}

// Code i of row `row` of a KVarN tile's code planes (rows of `len` codes: 256 for K's token
// rows, 128 for V's channel rows).
KVQ_HD int kvarn_code(const uint8_t* tile, int bits, int len, int row, int i) {
    int w[2];
    const int np = kvarn_planes(bits, w);
    int code = 0, s = 0;
    const uint8_t* plane = tile;
    for (int k = 0; k < np; ++k) {
        const int per = 8 / w[k];
        const uint8_t byte = plane[(int64_t)row * (len / per) + i / per];
        code |= ((byte >> (w[k] * (i % per))) & ((1 << w[k]) - 1)) << s;
        s += w[k];
        plane += 4096 * w[k];
    }
    return code;
}

// The 32-value block formats beyond Q8_0 / Q4_0: code bits (0 for any other format), the
// symmetric level count L (_0: codes x/d + L + 1) or 0 for the min-offset formats (_1: codes
// (x - m)/d in 0..2^bits - 1). Their records are token-major for K and V: the low nibble plane
// [128][D/2], the high plane (5-bit codes: one bit [128][D/8]; 6-bit: two bits [128][D/4]),
// d [128][D/32] fp16, then for the _1 formats m [128][D/32] fp16.
KVQ_HD int qblock_bits(int fmt) {
    switch (fmt) {
        case KVQ_Q5_0: return 5;
        case KVQ_Q6_0: return 6;
        case KVQ_Q4_1: return 4;
        case KVQ_Q5_1: return 5;
        default: return 0;
    }
}
KVQ_HD int qblock_sym_levels(int fmt) { return fmt == KVQ_Q5_0 ? 15 : (fmt == KVQ_Q6_0 ? 31 : 0); }

// Record bytes of one 128-position group of one KV head (K or V), per format.
KVQ_HD int64_t record_bytes(int fmt, int D) {
    switch (fmt) {
        case KVQ_TBQ4: return 66LL * D;                       // 64 B idx + 2 B norm per 128
        case KVQ_Q8_0: return 136LL * D;                      // 34 B per 32, 128 tokens
        case KVQ_Q4_0: return 72LL * D;                       // 18 B per 32
        case KVQ_Q5_0: return 88LL * D;                       // 22 B per 32
        case KVQ_Q6_0: return 104LL * D;                      // 26 B per 32
        case KVQ_Q4_1: return 80LL * D;                       // 20 B per 32
        case KVQ_Q5_1: return 96LL * D;                       // 24 B per 32
        case KVQ_TURBO3: return 50LL * D;                     // 48 B idx + 2 B norm per 128
        case KVQ_TQ5_0: return 82LL * D;                      // 80 B codes + 2 B scale per 128
        case KVQ_KVARN2: case KVQ_KVARN3: case KVQ_KVARN4: case KVQ_KVARN5: case KVQ_KVARN6: case KVQ_KVARN8:
            return (int64_t)(D / 256) * (4096 * kvarn_bits(fmt) + 1152);
        default: return -1;
    }
}

// Code bytes (before the scale area) of a non-KVarN record.
KVQ_HD int64_t record_code_bytes(int fmt, int D) {
    switch (fmt) {
        case KVQ_TBQ4: return 64LL * D;
        case KVQ_Q8_0: return 128LL * D;
        case KVQ_Q4_0: return 64LL * D;
        case KVQ_Q5_0: case KVQ_Q5_1: return 80LL * D;       // nibbles + one-bit plane
        case KVQ_Q6_0: return 96LL * D;                       // nibbles + two-bit plane
        case KVQ_Q4_1: return 64LL * D;
        case KVQ_TURBO3: return 48LL * D;                     // 2-bit plane + one-bit plane
        case KVQ_TQ5_0: return 80LL * D;                      // nibbles + one-bit plane
        default: return -1;
    }
}

KVQ_HD int rotation_of(int fmt) {
    if (fmt == KVQ_TBQ4 || fmt == KVQ_TURBO3 || fmt == KVQ_TQ5_0) return ROT_TBQ128;
    if (kvarn_bits(fmt)) return ROT_HAD256;
    return ROT_NONE;
}

KVQ_HD int64_t align256(int64_t x) { return (x + 255) & ~(int64_t)255; }

// Geometry of the device pool. Every per-(layer, seq, head) region of kind X for
// which w (0 = K, 1 = V) lives at  base + off_X[w] + unit * stride_X[w]  with
// unit = (layer * max_seqs + seq) * H + head.
struct Layout {
    int32_t L, H, D, Hq, G, NQ;
    int32_t max_seqs, T, R, gcap;
    int64_t max_ctx;
    int32_t fmt[2];          // body format of K, V
    int32_t journal, tail_fmt, rot, jrow_bytes;   // jrow_bytes: bytes of one journal code row
    float scale;             // softmax scale
    int32_t kvarn_best;      // KVarN seals: 1 = 8 passes keeping the best state, 0 = 16 passes
    int64_t status_off;
    int64_t sink_off[2], sink_stride[2];
    int64_t jcode_off[2], jcode_stride[2];
    int64_t jscale_off[2], jscale_stride[2];
    int64_t tail_off[2], tail_stride[2];
    int64_t body_off[2], body_stride[2], rec_bytes[2];
    int64_t total;

    KVQ_HD int64_t unit(int l, int s, int h) const { return ((int64_t)l * max_seqs + s) * H + h; }
};

// Builds the layout; returns false on an invalid config (host side).
bool make_layout(const kvq_config& c, Layout* out);

// ---------------------------------------------------------------------------- launches
// One contiguous span of positions of one sequence that the decode kernel reads with a
// single region reader.
enum RegionKind : int32_t { RK_SINK = 0, RK_BODY = 1, RK_RING = 2, RK_TAIL = 3, RK_JEXACT = 4 };

struct SeqSpan {
    int32_t slot;            // sequence slot in the pool
    int32_t n_tok;           // N
    int32_t lo[4], hi[4];    // region-kernel spans in read order (sink, [body], ring span or exact journal, tail)
    int32_t kind[4];         // RegionKind of each span
    int32_t nchunk[4];       // chunks of each span
    int32_t items_per_head;  // region work items per KV head (sum of nchunk)
    int32_t first_item;      // index of this sequence's first region work item
    int32_t body_groups;     // sealed groups [128, S)
    int32_t body_per_head;   // body work items per KV head
    int32_t body_first;      // index of this sequence's first body work item
};

struct AttnParams {
    const void* pool;
    const uint16_t* q;       // [n_seq][Hq][D] fp16
    uint16_t* out;           // [n_seq][Hq][D] fp16
    float* partials;         // workspace: per item [2 * NQ + NQ * D] floats
    // fused decode step: the newest position's K and V rows ([n_seq][H][D] fp16, appended by
    // the region item that holds that position, which also reads them from here), else null
    const uint16_t* knew;
    const uint16_t* vnew;
    int32_t layer, n_seq, chunk, total_items;
    int32_t n_region_items;  // region items come first, body items after them
    int32_t ring_chunk;      // positions per region item of a tq6_0 ring span (others: chunk)
    int32_t region_first;    // the streaming kernel's first blocks take the region items (else the body items)
    // 1: the launch ahead in the stream is the merge kernel of the previous layer of the same
    // decode step, which lets this launch start once every launch before it has completed. The
    // items then read the cache and the step's inputs at once (nothing the merge writes) and
    // wait for the merge only before writing their partials (the buffer it is reading).
    int32_t early;
    SeqSpan seq[kMaxSeqPerCall];
};

struct AppendParams {
    const void* pool;
    const uint16_t* k;       // [n_seq][src_stride][H][D]
    const uint16_t* v;
    int32_t layer, n_seq, n_tok, src_stride;   // n_tok: the largest count; src_stride: input rows per sequence
    int32_t slot[kMaxSeqPerCall];
    int32_t n0[kMaxSeqPerCall];       // N before this append
    int32_t count[kMaxSeqPerCall];    // positions appended to this sequence (<= n_tok)
    int32_t src_off[kMaxSeqPerCall];  // input row of position n0
    int32_t tail_from[kMaxSeqPerCall];   // positions >= tail_from also write the exact tail
};

struct SealSeq {             // one sequence's batch of consecutive groups (same in every sealed layer)
    int32_t slot;
    int32_t first_pos;       // position of the first group to seal
    int32_t first_group;     // its body group index
    int32_t n_groups;
    int32_t prefix;          // groups of the earlier sequences of this launch
    int32_t pad;
    int64_t src_row;         // input source: input row of first_pos ([n_seq][src_stride][H][D])
};

struct SealParams {
    const void* pool;
    // input source (a prefill chunk sealed straight from the caller's fp16 rows), else null: the
    // rows come from the journal
    const uint16_t* k_src;
    const uint16_t* v_src;
    int32_t layer0, n_layers, n_seq, groups_per_layer;
    int32_t src_stride, pad;
    SealSeq seq[kMaxSeqPerCall];
};

// Device constants: TBQ4 centroids / boundaries and sign vectors (host-derived).
struct FormatTables {
    float cent[16];
    float bnd[15];
    float pad;
    uint64_t sign_words[4];
    float cent3[8];        // turbo3: 8-level table
    float bnd3[7];
    float pad3;
};

const FormatTables& host_tables();   // derived once per process (tables.cpp)

// Kernel launchers (kernels_*.cu). Each returns cudaError_t as int.
int launch_append(const Layout& lay, const AppendParams& p, void* stream);
int launch_seal(const Layout& lay, const SealParams& p, void* stream);
int launch_seal_rows(const Layout& lay, const SealParams& p, void* stream);   // TBQ4 / Q8_0 / Q4_0
// Events recorded around the decode kernel's launch (both null: none); flags for
// cudaEventRecordWithFlags (cudaEventRecordExternal while a graph is captured).
struct LaunchMarks {
    void* before = nullptr;
    void* after = nullptr;
    unsigned flags = 0;
    bool pdl = false;      // launch the decode and merge kernels with programmatic stream serialization
    bool early = false;    // with pdl: the launch ahead is this step's previous merge (AttnParams::early)
    // with side (a stream joined to the capture) and fork (an event) set, each mark is recorded
    // on the side stream after a fork from the launching stream, so no event node sits between
    // two kernels and their programmatic launch stays in place
    void* side = nullptr;
    void* fork = nullptr;
};
int launch_decode(const Layout& lay, const AttnParams& p, void* stream, const LaunchMarks& marks = LaunchMarks());
int launch_decode_fused(const Layout& lay, const AttnParams& p, int n_body, int n_region, void* stream,
                        bool pdl = false);
int upload_tables_body(const FormatTables& t);
int launch_wait_probe(const Layout& lay, const void* pool, uint64_t limit_ns, void* stream);
int body_ctas_per_sm(const Layout& lay);     // resident body-item CTAs per SM (0: no instance)
int decode_ctas_per_sm(const Layout& lay);   // the same with the region items in the kernel
int region_kernel_ok(const Layout& lay);     // 1 if the streaming kernel takes the region items
int launch_dequant(const Layout& lay, const void* pool, int layer, int slot, int head, int which,
                   int kind, int64_t p0, int64_t n, float* out, void* stream);
int upload_tables_codec(const FormatTables& t);
int upload_tables_seal(const FormatTables& t);
const kvq_config* cache_config(const kvq_cache* c);   // the config a handle was created with
int upload_tables_attn(const FormatTables& t);
int query_sm_count(int device);

}  // namespace kvq
