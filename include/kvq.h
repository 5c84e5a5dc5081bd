/*
 * kvq.h — C ABI of the rotated low-bit KV cache and its decode attention (GB300, sm_103a).
 *
 * The calls mirror how the source pages state the problem: a KV cache written one token
 * at a time into a staging journal (SJ-KVaRN §2.1 "The life of a token"), sealed in
 * batches into compact body records (SJ-KVaRN §2.1 item 4, §4.3 "Adaptive tail"), read by
 * one decode-attention pass that merges every region under one softmax (KV Cache
 * Precision Tail §2; HAL #582 §5 P2, the two-region streaming combine), and sized in
 * bytes per token (KV cache math, "Bytes per token").
 *
 * Conventions for every call:
 *  - Return value: a kvq_status. No call throws or aborts across the ABI.
 *  - Device pointers are plain CUDA device addresses, 16-byte aligned; host pointers are
 *    plain host addresses. Nothing here takes or returns framework (torch) types.
 *  - Ownership: the caller allocates the device pool, the decode workspace and every input
 *    and output buffer. The library keeps only host-side metadata (an opaque kvq_cache)
 *    plus pointers into the caller's pool, and never calls cudaMalloc.
 *  - Ordering: device work is enqueued on the given stream (cudaStream_t passed as void*;
 *    NULL is the legacy default stream). Lengths live on the host and are authoritative,
 *    so refusals (KVQ_ENOSPC, KVQ_EINVAL) happen before anything is enqueued.
 *  - Errors detected on the device (non-finite scales: bit 0; a bounded wait that ran
 *    out: bit 1) set bits of a status word that kv_get_status reads after the caller
 *    synchronises.
 *
 * Shapes: L layers, H KV heads, Hq query heads, G = Hq / H, D head_dim. Query head h reads
 * KV head h / G. K/V/q inputs are IEEE fp16, row-major.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVQ_OK = 0,
    KVQ_EINVAL = 1,        /* bad argument: null / misaligned pointer, index out of range, bad config */
    KVQ_ENOSPC = 2,        /* journal ring or context capacity would overflow; nothing written */
    KVQ_EUNSUPPORTED = 3,  /* valid config this library has no kernel for */
    KVQ_ECUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    KVQ_EDEVICE = 5        /* device status word reports a problem (see kv_get_status) */
} kvq_status;

/* Stored formats. Body formats: TBQ4, TURBO3, TQ5_0, Q8_0, Q4_0, Q5_0, Q6_0, Q4_1, Q5_1,
 * KVARN2..KVARN8.
 * Journal: TQ6_0, F16, BF16.
 * Exact tail: F16, BF16. K and V bodies may differ (e.g. KVARN3 keys, KVARN2 values). */
typedef enum {
    KVQ_F16 = 0,
    KVQ_BF16 = 1,
    KVQ_TQ6_0 = 2,   /* SJ-KVaRN §2.1: rotated 6-bit, 98 B per 128 values */
    KVQ_TBQ4 = 3,    /* KV cache math: sign flip, WHT, sign flip; 16 Lloyd-Max centroids; 66 B/128 */
    KVQ_Q8_0 = 4,    /* 34 B per 32 values */
    KVQ_Q4_0 = 5,    /* 18 B per 32 values */
    KVQ_KVARN4 = 6,  /* SJ-KVaRN §2.2: 256-pt Hadamard, 16-pass balancing, 4-bit rows */
    KVQ_KVARN5 = 7,  /* same, 5-bit rows */
    KVQ_KVARN2 = 8,  /* same, 2-bit rows (SJ-KVaRN §2.3 scalar body, §3: the 3/2 and 2/2 caches) */
    KVQ_KVARN3 = 9,  /* same, 3-bit rows */
    KVQ_KVARN6 = 10, /* same, 6-bit rows */
    KVQ_KVARN8 = 11, /* same, 8-bit rows (KVarN8, the pages' ceiling check) */
    /* 32-value block formats the pages compare against (SJ-KVaRN §4.1, §6; the Qwen page):
     * symmetric d = fp16(max|x| / L) with codes x/d + L + 1, or the block minimum as offset
     * m = fp16(min x), d = fp16((max - min) / Q), codes (x - m)/d. Records token-major for K and V. */
    KVQ_Q5_0 = 12,   /* L = 15: 22 B per 32 values */
    KVQ_Q6_0 = 13,   /* L = 31: 26 B per 32 values */
    KVQ_Q4_1 = 14,   /* Q = 15: 20 B per 32 values */
    KVQ_Q5_1 = 15,   /* Q = 31: 24 B per 32 values */
    /* rotated comparators of the pages (SJ-KVaRN §2.1, §4.1; KV cache math), TBQ4's rotation:
     * turbo3 = TBQ with the 8-level Lloyd-Max table (fp16 norm + 3-bit indices, 50 B per 128);
     * tq5_0 = symmetric 5-bit, d = fp16(max|y| / 15) (82 B per 128). Records token-major. */
    KVQ_TURBO3 = 16,
    KVQ_TQ5_0 = 17
} kvq_fmt;

/* Balancing rule of KVarN seals (SJ-KVaRN §2.2 "Rotation and balancing"): 16 alternating
 * row/column passes keeping the final scales, or the KVarN reference configuration's 8 passes
 * keeping the best scales seen. Reading of "best": the state whose largest |sigma - 1| over
 * the lines the last pass did not balance (the columns after a row pass, the rows after a
 * column pass; sigma the line's spread as the next pass would compute it) is the smallest,
 * the earliest pass on a tie. Records have the same layout either way. */
enum { KVQ_KVARN_FINAL16 = 0, KVQ_KVARN_BEST8 = 1 };

typedef struct {
    int32_t n_layers;
    int32_t n_kv_heads;
    int32_t head_dim;        /* 128, 256 or 512; KVarN bodies need a multiple of 256 */
    int32_t n_q_heads;       /* a multiple of n_kv_heads, with n_q_heads / n_kv_heads <= 16 */
    int32_t max_seqs;        /* sequence slots */
    int32_t kvarn_balance;   /* KVarN bodies: KVQ_KVARN_FINAL16 (0) or KVQ_KVARN_BEST8 (1) */
    int64_t max_ctx;         /* positions a slot can hold (sets the body capacity) */
    int32_t k_body;          /* kvq_fmt of K body records */
    int32_t v_body;          /* kvq_fmt of V body records; must share K's rotation */
    int32_t journal;         /* KVQ_TQ6_0 (rotated ring + exact tail) or KVQ_F16 / KVQ_BF16 */
    int32_t tail_fmt;        /* exact store format, KVQ_F16 or KVQ_BF16 (equals journal when exact) */
    int32_t tail;            /* T: exact tail positions; also the smallest allowed seal keep */
    int32_t ring_capacity;   /* R: journal positions, a multiple of 128 */
    float softmax_scale;     /* 0 selects 1/sqrt(head_dim) */
    int32_t reserved1;
} kvq_config;

/* Byte accounting (KV cache math, "Bytes per token"; SJ-KVaRN §3 and §7.2). All figures
 * cover every layer and KV head, K and V together. */
typedef struct {
    int64_t body_bytes_per_token;    /* compact body records */
    int64_t f16_bytes_per_token;     /* the same shape at 16 bits: 2 x L x H x D x 2 */
    int64_t journal_bytes_per_slot;  /* one journal ring position */
    int64_t tail_bytes_per_slot;     /* one exact-tail position (0 without a tq6_0 journal) */
    int64_t sink_bytes;              /* the 128-position sink of one sequence */
    int64_t fixed_bytes_per_seq;     /* sink + full journal ring + tail of one sequence */
    int64_t pool_bytes;              /* device pool kv_create needs for this config */
} kvq_bytes;

typedef struct kvq_cache kvq_cache;  /* opaque host-side handle */

/* kv_bytes_per_token — closed-form sizes of a config (KV cache math, "Bytes per token":
 * 2 x layers x KV heads x head_dim x bytes per value; block formats by block bytes).
 * Pure host arithmetic; out is a host pointer. KVQ_EINVAL on a bad config. */
kvq_status kv_bytes_per_token(const kvq_config* cfg, kvq_bytes* out);

/* kv_auto_tier — the least compression that keeps a whole cache of `tokens` positions inside
 * `budget_bytes` (HAL #582 §5 P1, "auto KV-tier policy at boot": walk the ladder f16 ->
 * q8_0 K / q8_0 V -> q8_0 K / q4_0 V -> q5_1 K / q4_0 V and take the first rung whose cost
 * fits; the floor rung, q5_1 / q4_0, when none does). A rung's cost is tokens x layers x KV
 * heads x head_dim x (bytes per K value + bytes per V value), the per-cell byte sum the page
 * budgets with (f16 2 B, q8_0 34/32 B, q5_1 24/32 B, q4_0 18/32 B per value). Reading: the f16
 * rung means an uncompressed cache (*k_fmt = *v_fmt = KVQ_F16: an F16 journal that holds the context,
 * never sealed). Only n_layers, n_kv_heads and head_dim of cfg are read. Host arithmetic,
 * host pointers out: the chosen formats and their cost in bytes. KVQ_OK when the chosen rung
 * fits, KVQ_ENOSPC with the floor rung when none fits, KVQ_EINVAL on a null pointer, a
 * non-positive shape or tokens < 0. */
kvq_status kv_auto_tier(const kvq_config* cfg, int64_t tokens, uint64_t budget_bytes, int32_t* k_fmt,
                        int32_t* v_fmt, uint64_t* cost_bytes);

/* kv_tier_budget — the cache budget of that policy (HAL #582 §5 P1): the device's free bytes,
 * capped by a total target (0: no target), less the bytes already resident and a 1.5 GiB
 * compute reserve; 0 when that is negative. Host arithmetic; budget is a host pointer.
 * KVQ_EINVAL on a null pointer. */
kvq_status kv_tier_budget(uint64_t free_bytes, uint64_t resident_bytes, uint64_t target_bytes, uint64_t* budget);

/* kv_required_bytes — device pool bytes for kv_create and workspace bytes for
 * kv_decode_attn with up to cfg->max_seqs sequences per call. Host pointers out. */
kvq_status kv_required_bytes(const kvq_config* cfg, size_t* pool_bytes, size_t* workspace_bytes);

/* kv_create — bind a config to a caller-owned device pool (>= pool_bytes from
 * kv_required_bytes, 256-byte aligned) on CUDA device `device`. Every slot starts empty
 * (N = 0, sealed end S = 128). Zeroes the pool's status word (synchronously). The handle
 * is freed by kv_destroy; the pool stays the caller's. */
kvq_status kv_create(const kvq_config* cfg, void* device_pool, size_t pool_bytes, int device,
                     kvq_cache** out);
kvq_status kv_destroy(kvq_cache* cache);

/* kv_reset — empty one slot of one layer (layer -1: all layers). Host metadata only. */
kvq_status kv_reset(kvq_cache* cache, int layer, int seq);

/* kv_append — SJ-KVaRN §2.1: write positions N..N+n_tok-1 of each listed sequence of one
 * layer. k, v: device fp16 [n_seq][n_tok][H][D]. Position p < 128 goes to the fp16 sink;
 * p >= 128 goes to the journal slot (p - 128) mod R — tq6_0 of the rotated vector, or a
 * verbatim F16 / round-to-nearest-even BF16 copy — and, with a tq6_0 journal, also to the
 * exact tail slot p mod T. seq_ids: host int32 [n_seq], distinct. KVQ_ENOSPC (no write)
 * if a journal would hold more than R unsealed positions or N would exceed max_ctx. */
kvq_status kv_append(kvq_cache* cache, int layer, const int32_t* seq_ids, int n_seq, int n_tok,
                     const void* k, const void* v, void* stream);

/* kv_prefill — a prefill chunk in one call (SJ-KVaRN §2.1: positions staged, then every full
 * group older than the newest `keep` committed in one batch): for each listed sequence of
 * `layer`, positions N..N+n_tok-1 from k / v ([n_seq][n_tok][H][D] fp16, device, as kv_append),
 * then the seal of every full group g with S + 128 <= N + n_tok - keep (as kv_seal). The cache
 * ends byte for byte as kv_append followed by kv_seal would leave it; a group that lies wholly in
 * the chunk and is sealed by this call is encoded straight from the input rows, through the
 * values the journal would have returned (bf16 rounding for a BF16 journal, the rotation, and
 * with a tq6_0 ring its quantize-dequantize), so it never occupies the journal: n_tok is bounded
 * by max_ctx, not by the ring. Refused with nothing written: KVQ_ENOSPC when N + n_tok exceeds
 * max_ctx or the positions the call leaves unsealed exceed ring_capacity; KVQ_EINVAL on a bad
 * layer, sequence list, keep < tail or null pointer. groups_sealed: host out (may be null). */
kvq_status kv_prefill(kvq_cache* cache, int layer, const int32_t* seq_ids, int n_seq, int n_tok, const void* k,
                      const void* v, int keep, int64_t* groups_sealed, void* stream);

/* kv_prefill_plan — (test call) the host plan kv_prefill makes for one sequence holding
 * n_tokens positions with sealed end sealed_end: ranges (host, 8 values) receives the head
 * [r0, r1) appended to the journal and sink, the groups [r2, r3) then sealed from the journal,
 * the groups [r4, r5) sealed straight from the input rows, and the rest [r6, r7) appended to the
 * journal and exact tail; r5 is the sealed end after the call. kv_prefill takes its counts,
 * offsets and rows from this same plan. The same refusals as kv_prefill (KVQ_ENOSPC); KVQ_EINVAL
 * on a null pointer, n_tok <= 0, or a sealed_end that is not 128 plus a multiple of 128. Pure
 * host arithmetic. */
kvq_status kv_prefill_plan(int64_t n_tokens, int64_t sealed_end, int64_t n_tok, int32_t keep, int32_t ring_capacity,
                           int64_t max_ctx, int64_t ranges[8]);

/* kv_seal — SJ-KVaRN §2.1 item 4 and §4.3: for each listed sequence of `layer` (-1: all
 * layers) seal every full 128-position group g with S + 128 <= N - keep into body records,
 * oldest first, and advance S. keep >= T. groups_sealed (host, may be NULL) receives the
 * number of (layer, sequence) groups sealed. The count is decided on the host before launch. */
kvq_status kv_seal(kvq_cache* cache, int layer, const int32_t* seq_ids, int n_seq, int keep,
                   int64_t* groups_sealed, void* stream);

/* kv_decode_attn — one decode step of attention for each listed sequence of one layer over
 * all N positions it holds: scores s_i = scale * <q, k_i> with the raw query on the exact
 * regions (sink, exact tail, exact journal) and the rotated query R q on the rotated regions
 * (body, tq6_0 ring span); one softmax over all positions; the rotated regions' weighted
 * sum rotated back once (KV cache math, "rotate first"; KV Cache Precision Tail §2).
 * q: device fp16 [n_seq][Hq][D]; out: device fp16 [n_seq][Hq][D].
 * workspace: device, >= workspace_bytes of kv_required_bytes. It holds the call's per-item
 * partials (m, l, o), each written before it is read, so its contents need not start at zero.
 * Calls sharing a workspace must not overlap on the GPU. */
kvq_status kv_decode_attn(kvq_cache* cache, int layer, const int32_t* seq_ids, int n_seq,
                          const void* q, void* out, void* workspace, size_t ws_bytes, void* stream);

/* kv_decode_step — one decode step over layers [0, n_layers) issued from C: for each layer
 * l, kv_append of one position per sequence, then kv_seal(l, keep) of the sequences whose
 * journal calls for it, then kv_decode_attn. Seal policy: seal_trigger > 0 seals a sequence
 * when its journal holds seal_trigger positions (SJ-KVaRN §4.3 adaptive tail: grow to 8,192,
 * seal back to the newest 4,096); seal_trigger == 0 seals whenever a full group older than
 * keep exists; seal_trigger < 0 never seals. Layouts: q [n_layers][n_seq][Hq][D], k and v
 * [n_layers][n_seq][1][H][D], out [n_layers][n_seq][Hq][D], all device fp16.
 * events (may be NULL): 2 * n_layers caller-created cudaEvent_t handles; events[2l]
 * completes when everything layer l's decode kernel waits for has completed, events[2l+1]
 * when that kernel (the streaming kernel, or the generic split kernel; the merge kernel
 * follows) has. In graph mode they are event-record nodes on a side branch of the step's
 * graph, so the kernels keep their programmatic launches; with graph mode off they are
 * recorded inline on `stream` and the decode and merge kernels are launched plainly.
 * groups_sealed (host, may be NULL) receives the groups sealed in this step.
 * Where the decode kernel takes a layout's region items and the newest row is fp16, the
 * append runs inside that layer's attention launch (same results, one launch less).
 * By default (kv_set_graph_mode) the step's launches are captured on a stream private to the
 * cache and replayed on `stream` as one CUDA graph; an argument or capacity error then leaves
 * the cache as it was (nothing launched). With graph mode off the calls go straight to
 * `stream`, and a failing call stops the step with earlier layers applied. */
kvq_status kv_decode_step(kvq_cache* cache, int n_layers, const int32_t* seq_ids, int n_seq,
                          const void* q, const void* k, const void* v, void* out,
                          int seal_trigger, int keep, void* workspace, size_t ws_bytes,
                          void* const* events, int64_t* groups_sealed, void* stream);

/* kv_set_graph_mode — whether kv_decode_step replays its launches as one CUDA graph (enable
 * != 0, the default) or issues them one by one. A step is launch-bound where its kernels are
 * short: on GB300 a dependent launch costs 2 to 4 us on a stream, about 1 us as a graph node.
 * The graph is re-captured each step and applied to the cached executable graph with
 * cudaGraphExecUpdate, instantiated anew when the launch topology changes (a seal, another
 * layer count). If a capture or a graph launch fails, the cache switches to direct launches.
 * A library convenience with no counterpart in the source pages. */
kvq_status kv_set_graph_mode(kvq_cache* cache, int enable);

/* kv_snapshot_size / kv_snapshot / kv_restore — copy the host-side lengths of every slot
 * out of, or back into, a cache handle (host memory of kv_snapshot_size bytes). Restoring
 * is valid only together with the device pool contents of the same moment; the caller owns
 * both copies. Used to replay a benchmark from one starting state. */
kvq_status kv_snapshot_size(const kvq_cache* cache, size_t* bytes);
kvq_status kv_snapshot(const kvq_cache* cache, void* buf, size_t bytes);
kvq_status kv_restore(kvq_cache* cache, const void* buf, size_t bytes);

/* kv_decode_attn_noalloc — kv_decode_attn for callers that cannot allocate device memory
 * (for example a host program that only links this ABI inside a runtime whose memory manager
 * already owns the device, or a loop that cannot afford cudaMalloc's implicit
 * synchronisation). The source pages have no counterpart: this is a library convenience.
 * Same arguments and results as kv_decode_attn, minus the workspace: the library uses a
 * fixed 32 MiB device array that every GPU loading the library holds until exit. Configs whose
 * kv_required_bytes workspace exceeds 32 MiB are refused with KVQ_EUNSUPPORTED. All calls
 * share the array (as with kv_decode_attn's workspace, nothing in it needs to start at zero:
 * every partial is written before it is read); calls that overlap on the GPU race
 * and must be avoided. The first call on each device looks up the array's address with that
 * device current; make that first call before any stream capture begins. Allocates nothing. */
kvq_status kv_decode_attn_noalloc(kvq_cache* cache, int layer, const int32_t* seq_ids, int n_seq,
                                  const void* q, void* out, void* stream);

/* kv_state — host copies of one slot's lengths. */
kvq_status kv_state(const kvq_cache* cache, int layer, int seq, int64_t* n_tokens, int64_t* sealed_end);

/* kv_get_status — read (synchronously) and clear the device status word. Bit 0: a
 * non-finite scale was produced by an encoder (the record holds it, as the format defines).
 * Bit 1: a bounded device wait (a streaming kernel's wait for its bulk copies, 2 s) ran out;
 * the outputs of the launch that set it are invalid. Returns KVQ_EDEVICE if any bit was set. */
kvq_status kv_get_status(kvq_cache* cache, uint32_t* word);

/* ---------------------------------------------------------------------------------------
 * Test and inspection calls (not on the decode path).
 * ------------------------------------------------------------------------------------- */

/* kv_dequant — decode positions [p0, p0+n) of (layer, seq, KV head, which: 0 = K, 1 = V)
 * from whichever region holds them, into device fp32 out [n][D]: sink/exact values as
 * stored, body and tq6_0 ring values in the rotated domain, with the format's dequant
 * arithmetic (bit-exact definition). Positions must lie in [0, N). */
kvq_status kv_dequant(kvq_cache* cache, int layer, int seq, int head, int which, int64_t p0,
                      int64_t n, float* out, void* stream);

/* kv_test_wait_timeout — (test call) exercises the streaming kernels' bounded-wait path: one
 * CTA waits on an mbarrier that no copy completes, with a limit of limit_ns (1 us .. 10 s) of
 * the GPU's global timer instead of the kernels' 2 s, then waits (2 s bound) for the one bulk
 * copy it did issue and retires. On return the wait has run out, so after the caller
 * synchronises, kv_get_status reports bit 1; the context stays usable. KVQ_EINVAL on a limit
 * out of range. A library test hook with no counterpart in the source pages. */
kvq_status kv_test_wait_timeout(kvq_cache* cache, uint64_t limit_ns, void* stream);

/* Region ids for kv_region_ptr. */
enum {
    KVQ_REGION_SINK = 0,        /* fp16 [128][D] */
    KVQ_REGION_JOURNAL = 1,     /* tq6_0: codes [R][D/128][96]; exact: [R][D] 16-bit */
    KVQ_REGION_JOURNAL_SCALE = 2, /* tq6_0 only: fp16 [R][D/128] */
    KVQ_REGION_TAIL = 3,        /* tq6_0 journal only: [T][D] 16-bit */
    KVQ_REGION_BODY = 4         /* records [capacity groups][record bytes] */
};

/* kv_region_ptr — device address and byte size of one region's storage for
 * (layer, seq, KV head, which). For inspection (byte-exact comparisons) only. */
kvq_status kv_region_ptr(const kvq_cache* cache, int layer, int seq, int head, int which,
                         int region, void** ptr, size_t* bytes);

/* kv_format_tables — the constants this library derived on its own at load time: the TBQ4
 * centroids and boundaries (fp32, Lloyd-Max for N(0, 1/128)) and the four splitmix64 sign
 * words. Host pointers; any may be NULL. */
kvq_status kv_format_tables(float centroids[16], float boundaries[15], uint64_t sign_words[4]);

/* kv_format_tables_turbo3 — turbo3's 8 centroids and 7 boundaries (fp32, the same Lloyd-Max
 * construction with 8 levels) as this library derived them. Host pointers; either may be NULL. */
kvq_status kv_format_tables_turbo3(float centroids[8], float boundaries[7]);

/* kv_status_string — static description of a status code. */
const char* kv_status_string(kvq_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
