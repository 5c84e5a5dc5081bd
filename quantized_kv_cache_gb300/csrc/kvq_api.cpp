// Host side of the C ABI (include/kvq.h): configuration checks, the device-pool layout,
// host-authoritative lengths, work decomposition and kernel launches. Lengths of every
// (layer, sequence) live here, so refusals happen before anything is enqueued, and the
// decode work list is derived from them without reading device memory.
#include <cuda_runtime.h>
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <vector>
#include "kvq_internal.h"
#include "../../include/kvq_synth.h"

using namespace kvq;

struct kvq_cache {
    kvq_config cfg;
    Layout lay;
    void* pool;
    size_t pool_bytes;
    int device;
    int sm_count;
    std::vector<int64_t> n_tok;   // [L][max_seqs]
    std::vector<int64_t> sealed;  // [L][max_seqs]
    // kv_decode_step replays its launches as one CUDA graph: captured on a private stream each
    // call and applied to the cached executable graph with cudaGraphExecUpdate (instantiated
    // anew when the launches' topology changes: a seal, another layer count)
    int graph_mode = 1;
    cudaStream_t cap_stream = nullptr;
    cudaGraphExec_t step_exec = nullptr;
    cudaStream_t mark_stream = nullptr;    // side branch of a captured step for the caller's events
    cudaEvent_t mark_fork = nullptr;
};

namespace kvq {

static bool is_body(int f) {
    return f == KVQ_TBQ4 || f == KVQ_TURBO3 || f == KVQ_TQ5_0 || f == KVQ_Q8_0 || f == KVQ_Q4_0 ||
           qblock_bits(f) != 0 || kvarn_bits(f) != 0;
}

bool make_layout(const kvq_config& c, Layout* out) {
    Layout L{};
    if (c.n_layers <= 0 || c.n_kv_heads <= 0 || c.max_seqs <= 0) return false;
    if (c.head_dim != 128 && c.head_dim != 256 && c.head_dim != 512) return false;
    if (c.n_q_heads <= 0 || c.n_q_heads % c.n_kv_heads) return false;
    const int G = c.n_q_heads / c.n_kv_heads;
    if (G > kMaxG) return false;
    if (!is_body(c.k_body) || !is_body(c.v_body)) return false;
    if (rotation_of(c.k_body) != rotation_of(c.v_body)) return false;
    if (rotation_of(c.k_body) == ROT_HAD256 && c.head_dim % 256) return false;
    if (c.journal != KVQ_TQ6_0 && c.journal != KVQ_F16 && c.journal != KVQ_BF16) return false;
    if (c.tail_fmt != KVQ_F16 && c.tail_fmt != KVQ_BF16) return false;
    if (c.journal != KVQ_TQ6_0 && c.tail_fmt != c.journal) return false;
    if (c.tail <= 0 || c.ring_capacity <= 0 || c.ring_capacity % kGroup) return false;
    if (c.ring_capacity < c.tail + kGroup) return false;   // a full group must fit beyond the tail
    if (c.max_ctx < kSink + kGroup || c.max_ctx > (int64_t)1 << 30) return false;
    if (!(c.softmax_scale >= 0.f) || !std::isfinite(c.softmax_scale)) return false;
    if (c.kvarn_balance != KVQ_KVARN_FINAL16 && c.kvarn_balance != KVQ_KVARN_BEST8) return false;
    L.L = c.n_layers; L.H = c.n_kv_heads; L.D = c.head_dim; L.Hq = c.n_q_heads; L.G = G;
    L.NQ = G <= 8 ? 8 : 16;
    L.max_seqs = c.max_seqs; L.T = c.tail; L.R = c.ring_capacity;
    L.gcap = (int32_t)((c.max_ctx - kSink + kGroup - 1) / kGroup);
    L.max_ctx = c.max_ctx;
    L.fmt[0] = c.k_body; L.fmt[1] = c.v_body;
    L.journal = c.journal; L.tail_fmt = c.tail_fmt; L.rot = rotation_of(c.k_body);
    L.jrow_bytes = (c.journal == KVQ_TQ6_0) ? (c.head_dim / 128) * 96 : c.head_dim * 2;
    L.scale = c.softmax_scale > 0.f ? c.softmax_scale : 1.0f / std::sqrt((float)c.head_dim);
    L.kvarn_best = c.kvarn_balance == KVQ_KVARN_BEST8 ? 1 : 0;
    const int64_t units = (int64_t)L.L * L.max_seqs * L.H;
    int64_t off = 256;   // status word area
    L.status_off = 0;
    auto region = [&](int64_t per_unit, int64_t* o, int64_t* st, int w) {
        st[w] = align256(per_unit);
        o[w] = off;
        off += st[w] * units;
    };
    for (int w = 0; w < 2; ++w) {
        region((int64_t)kSink * L.D * 2, L.sink_off, L.sink_stride, w);
        region((int64_t)L.R * L.jrow_bytes, L.jcode_off, L.jcode_stride, w);
        if (c.journal == KVQ_TQ6_0) {
            region((int64_t)L.R * (L.D / 128) * 2, L.jscale_off, L.jscale_stride, w);
            region((int64_t)L.T * L.D * 2, L.tail_off, L.tail_stride, w);
        }
        L.rec_bytes[w] = record_bytes(L.fmt[w], L.D);
        region((int64_t)L.gcap * L.rec_bytes[w], L.body_off, L.body_stride, w);
    }
    L.total = off;
    *out = L;
    return true;
}

const kvq_config* cache_config(const kvq_cache* c) { return c ? &c->cfg : nullptr; }

}  // namespace kvq

namespace {

std::mutex g_tab_mu;
std::set<int> g_tab_devices;

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

kvq_status ensure_tables(int device) {
    std::lock_guard<std::mutex> lk(g_tab_mu);
    if (g_tab_devices.count(device)) return KVQ_OK;
    const FormatTables& t = host_tables();
    if (upload_tables_codec(t) != 0 || upload_tables_seal(t) != 0 || upload_tables_attn(t) != 0 || upload_tables_body(t) != 0) return KVQ_ECUDA;
    g_tab_devices.insert(device);
    return KVQ_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

kvq_status check_cache(const kvq_cache* c) {
    if (!c) return KVQ_EINVAL;
    if (current_device() != c->device) return KVQ_EINVAL;
    return KVQ_OK;
}

kvq_status check_seqs(const kvq_cache* c, const int32_t* seq_ids, int n_seq) {
    if (!seq_ids || n_seq <= 0 || n_seq > kMaxSeqPerCall) return n_seq > kMaxSeqPerCall ? KVQ_EUNSUPPORTED : KVQ_EINVAL;
    for (int i = 0; i < n_seq; ++i) {
        if (seq_ids[i] < 0 || seq_ids[i] >= c->cfg.max_seqs) return KVQ_EINVAL;
        for (int j = 0; j < i; ++j)
            if (seq_ids[j] == seq_ids[i]) return KVQ_EINVAL;
    }
    return KVQ_OK;
}

int64_t& NT(kvq_cache* c, int l, int s) { return c->n_tok[(size_t)l * c->cfg.max_seqs + s]; }
int64_t& ST(kvq_cache* c, int l, int s) { return c->sealed[(size_t)l * c->cfg.max_seqs + s]; }

kvq_status cuda_status(int e) { return e == 0 ? KVQ_OK : KVQ_ECUDA; }

size_t workspace_items(const kvq_config& c) {
    const int n = std::min(c.max_seqs, kMaxSeqPerCall);
    return 2048 + (size_t)4 * c.n_kv_heads * n;
}

// Region-kernel spans of one sequence in read order: the sink, the body [128, S) when
// with_body (layouts the body kernel has no instance for), the ring span or exact journal,
// and the exact tail.
int spans(const Layout& L, int64_t N, int64_t S, int32_t lo[4], int32_t hi[4], int32_t kind[4], bool with_body) {
    int n = 0;
    auto add = [&](int64_t a, int64_t b, int k) {
        if (b > a) { lo[n] = (int32_t)a; hi[n] = (int32_t)b; kind[n] = k; ++n; }
    };
    add(0, std::min<int64_t>(N, kSink), RK_SINK);
    if (with_body) add(kSink, S, RK_BODY);
    if (L.journal == KVQ_TQ6_0) {
        const int64_t E = std::max<int64_t>(S, N - L.T);
        add(S, E, RK_RING);
        add(std::max<int64_t>(E, kSink), N, RK_TAIL);
    } else {
        add(std::max<int64_t>(S, kSink), N, RK_JEXACT);
    }
    for (int i = n; i < 4; ++i) { lo[i] = hi[i] = 0; kind[i] = 0; }
    return n;
}

}  // namespace

extern "C" {

const char* kv_status_string(kvq_status s) {
    switch (s) {
        case KVQ_OK: return "ok";
        case KVQ_EINVAL: return "invalid argument";
        case KVQ_ENOSPC: return "journal or context capacity exceeded";
        case KVQ_EUNSUPPORTED: return "unsupported configuration";
        case KVQ_ECUDA: return "CUDA error";
        case KVQ_EDEVICE: return "device status word set";
    }
    return "unknown status";
}

kvq_status kv_bytes_per_token(const kvq_config* cfg, kvq_bytes* out) {
    if (!cfg || !out) return KVQ_EINVAL;
    Layout L;
    if (!make_layout(*cfg, &L)) return KVQ_EINVAL;
    const int64_t LH = (int64_t)L.L * L.H;
    kvq_bytes b{};
    b.body_bytes_per_token = LH * (L.rec_bytes[0] + L.rec_bytes[1]) / kGroup;
    b.f16_bytes_per_token = 2 * LH * L.D * 2;
    b.journal_bytes_per_slot = 2 * LH * (cfg->journal == KVQ_TQ6_0 ? (int64_t)(L.D / 128) * 98 : (int64_t)L.D * 2);
    b.tail_bytes_per_slot = cfg->journal == KVQ_TQ6_0 ? 2 * LH * L.D * 2 : 0;
    b.sink_bytes = 2 * LH * kSink * L.D * 2;
    b.fixed_bytes_per_seq = b.sink_bytes + b.journal_bytes_per_slot * L.R + b.tail_bytes_per_slot * L.T;
    b.pool_bytes = L.total;
    *out = b;
    return KVQ_OK;
}

kvq_status kv_auto_tier(const kvq_config* cfg, int64_t tokens, uint64_t budget_bytes, int32_t* k_fmt,
                        int32_t* v_fmt, uint64_t* cost_bytes) {
    if (!cfg || !k_fmt || !v_fmt || !cost_bytes || tokens < 0) return KVQ_EINVAL;
    if (cfg->n_layers <= 0 || cfg->n_kv_heads <= 0 || cfg->head_dim <= 0) return KVQ_EINVAL;
    // bytes per 32 values of each rung's K and V format: f16 64, q8_0 34, q5_1 24, q4_0 18
    struct Rung { int32_t k, v; uint64_t k32, v32; };
    static const Rung ladder[] = {{KVQ_F16, KVQ_F16, 64, 64}, {KVQ_Q8_0, KVQ_Q8_0, 34, 34},
                                  {KVQ_Q8_0, KVQ_Q4_0, 34, 18}, {KVQ_Q5_1, KVQ_Q4_0, 24, 18}};
    const uint64_t cells = (uint64_t)tokens * (uint64_t)cfg->n_layers * (uint64_t)cfg->n_kv_heads *
                           (uint64_t)cfg->head_dim;   // values per K (and per V)
    const int n = (int)(sizeof(ladder) / sizeof(ladder[0]));
    for (int i = 0; i < n; ++i) {
        const uint64_t cost = cells / 32 * (ladder[i].k32 + ladder[i].v32) +
                              cells % 32 * (ladder[i].k32 + ladder[i].v32) / 32;
        *k_fmt = ladder[i].k;
        *v_fmt = ladder[i].v;
        *cost_bytes = cost;
        if (cost <= budget_bytes) return KVQ_OK;
    }
    return KVQ_ENOSPC;   // the floor rung, which does not fit either
}

kvq_status kv_tier_budget(uint64_t free_bytes, uint64_t resident_bytes, uint64_t target_bytes, uint64_t* budget) {
    if (!budget) return KVQ_EINVAL;
    constexpr uint64_t kReserve = 3ull << 29;   // 1.5 GiB compute reserve
    const uint64_t cap = (target_bytes > 0 && target_bytes < free_bytes) ? target_bytes : free_bytes;
    const uint64_t used = resident_bytes + kReserve;
    *budget = cap > used ? cap - used : 0;
    return KVQ_OK;
}

kvq_status kv_required_bytes(const kvq_config* cfg, size_t* pool_bytes, size_t* workspace_bytes) {
    if (!cfg) return KVQ_EINVAL;
    Layout L;
    if (!make_layout(*cfg, &L)) return KVQ_EINVAL;
    if (pool_bytes) *pool_bytes = (size_t)L.total;
    if (workspace_bytes) *workspace_bytes = workspace_items(*cfg) * (2 * L.NQ + (size_t)L.NQ * L.D) * sizeof(float);
    return KVQ_OK;
}

kvq_status kv_create(const kvq_config* cfg, void* device_pool, size_t pool_bytes, int device, kvq_cache** out) {
    if (!cfg || !out || !device_pool) return KVQ_EINVAL;
    Layout L;
    if (!make_layout(*cfg, &L)) return KVQ_EINVAL;
    if (pool_bytes < (size_t)L.total || ((uintptr_t)device_pool & 255)) return KVQ_EINVAL;
    if (current_device() != device) return KVQ_EINVAL;
    kvq_status st = ensure_tables(device);
    if (st != KVQ_OK) return st;
    if (cudaMemset(device_pool, 0, 256) != cudaSuccess) return KVQ_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return KVQ_ECUDA;
    kvq_cache* c = new kvq_cache;
    c->cfg = *cfg;
    c->lay = L;
    c->pool = device_pool;
    c->pool_bytes = pool_bytes;
    c->device = device;
    c->sm_count = sms;
    c->n_tok.assign((size_t)L.L * cfg->max_seqs, 0);
    c->sealed.assign((size_t)L.L * cfg->max_seqs, kSink);
    *out = c;
    return KVQ_OK;
}

kvq_status kv_destroy(kvq_cache* c) {
    if (!c) return KVQ_EINVAL;
    if (c->step_exec) cudaGraphExecDestroy(c->step_exec);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    if (c->mark_stream) cudaStreamDestroy(c->mark_stream);
    if (c->mark_fork) cudaEventDestroy(c->mark_fork);
    delete c;
    return KVQ_OK;
}

kvq_status kv_reset(kvq_cache* c, int layer, int seq) {
    if (!c || seq < 0 || seq >= c->cfg.max_seqs || layer < -1 || layer >= c->cfg.n_layers) return KVQ_EINVAL;
    for (int l = 0; l < c->cfg.n_layers; ++l) {
        if (layer >= 0 && l != layer) continue;
        NT(c, l, seq) = 0;
        ST(c, l, seq) = kSink;
    }
    return KVQ_OK;
}

kvq_status kv_append(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq, int n_tok,
                     const void* k, const void* v, void* stream) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (layer < 0 || layer >= c->cfg.n_layers || n_tok <= 0 || !k || !v || !aligned16(k) || !aligned16(v))
        return KVQ_EINVAL;
    if ((st = check_seqs(c, seq_ids, n_seq)) != KVQ_OK) return st;
    if ((int64_t)n_seq * n_tok > (int64_t)1 << 31) return KVQ_EINVAL;
    AppendParams p{};
    p.pool = c->pool;
    p.k = (const uint16_t*)k;
    p.v = (const uint16_t*)v;
    p.layer = layer;
    p.n_seq = n_seq;
    p.n_tok = n_tok;
    p.src_stride = n_tok;
    for (int i = 0; i < n_seq; ++i) {
        const int s = seq_ids[i];
        const int64_t N = NT(c, layer, s), S = ST(c, layer, s);
        if (N + n_tok > c->cfg.max_ctx) return KVQ_ENOSPC;
        if (std::max<int64_t>(N + n_tok, kSink) - S > c->cfg.ring_capacity) return KVQ_ENOSPC;
        p.slot[i] = s;
        p.n0[i] = (int32_t)N;
        p.count[i] = n_tok;
        p.src_off[i] = 0;
        p.tail_from[i] = (int32_t)(N + n_tok - c->cfg.tail);
    }
    const int e = launch_append(c->lay, p, stream);
    if (e != 0) return KVQ_ECUDA;
    for (int i = 0; i < n_seq; ++i) NT(c, layer, seq_ids[i]) += n_tok;
    return KVQ_OK;
}

namespace {

// Seals counts[i] groups of each listed sequence of one layer, from its sealed end on: from the
// journal (k_src null) or from input rows (src_row[i]: the input row of the first group's first
// position; the input holds src_stride rows per sequence). Advances the sealed ends.
int seal_counts(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq, const int64_t* counts,
                const void* k_src, const void* v_src, int src_stride, const int64_t* src_row, void* stream) {
    SealParams p{};
    p.pool = c->pool;
    p.k_src = (const uint16_t*)k_src;
    p.v_src = (const uint16_t*)v_src;
    p.layer0 = layer;
    p.n_layers = 1;
    p.src_stride = src_stride;
    int32_t acc = 0;
    for (int i = 0; i < n_seq; ++i) {
        if (counts[i] <= 0) continue;
        const int s = seq_ids[i];
        SealSeq& q = p.seq[p.n_seq++];
        q.slot = s;
        q.first_pos = (int32_t)ST(c, layer, s);
        q.first_group = (int32_t)((ST(c, layer, s) - kSink) / kGroup);
        q.n_groups = (int32_t)counts[i];
        q.prefix = acc;
        q.src_row = src_row ? src_row[i] : 0;
        acc += (int32_t)counts[i];
    }
    p.groups_per_layer = acc;
    if (acc == 0) return 0;
    const int e = launch_seal(c->lay, p, stream);
    if (e != 0) return e;
    for (int i = 0; i < n_seq; ++i)
        if (counts[i] > 0) ST(c, layer, seq_ids[i]) += (int64_t)kGroup * counts[i];
    return 0;
}

// Appends, for each listed sequence, count[i] positions from its N on, read from input rows
// src_off[i] on (src_stride rows per sequence); positions >= tail_from[i] also write the tail.
int append_ranges(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq, const void* k, const void* v,
                  int src_stride, const int64_t* count, const int64_t* src_off, const int64_t* tail_from,
                  void* stream) {
    AppendParams p{};
    p.pool = c->pool;
    p.k = (const uint16_t*)k;
    p.v = (const uint16_t*)v;
    p.layer = layer;
    p.n_seq = n_seq;
    p.src_stride = src_stride;
    int64_t most = 0;
    for (int i = 0; i < n_seq; ++i) {
        p.slot[i] = seq_ids[i];
        p.n0[i] = (int32_t)NT(c, layer, seq_ids[i]);
        p.count[i] = (int32_t)count[i];
        p.src_off[i] = (int32_t)src_off[i];
        p.tail_from[i] = (int32_t)std::min<int64_t>(tail_from[i], 0x7fffffff);
        most = std::max(most, count[i]);
    }
    if (most == 0) return 0;
    p.n_tok = (int32_t)most;
    const int e = launch_append(c->lay, p, stream);
    if (e != 0) return e;
    for (int i = 0; i < n_seq; ++i) NT(c, layer, seq_ids[i]) += count[i];
    return 0;
}

}  // namespace

namespace {
// One sequence's prefill plan: N0 positions held, S0 sealed end (a group boundary), n_tok new
// positions. r receives the eight bounds kv_prefill works with: the head [r0, r1) appended to the
// journal and sink, the groups [r2, r3) then sealed from the journal, the groups [r4, r5) sealed
// straight from the input rows (r5 = S1, the sealed end after the call: every full group older
// than the newest keep sealed), and the rest [r6, r7) appended to the journal and exact tail.
// With M = min(first group start >= N0, S1, N1): r1 = max(N0, M); r3 = r4 = the journal seal's
// end. KVQ_ENOSPC when the call would pass max_ctx or leave more unsealed positions than the
// ring holds.
kvq_status prefill_plan(int64_t N0, int64_t S0, int64_t n_tok, int64_t keep, int64_t R, int64_t max_ctx,
                        int64_t r[8]) {
    const int64_t N1 = N0 + n_tok;
    if (N1 > max_ctx) return KVQ_ENOSPC;
    const int64_t lim = N1 - keep - S0;
    const int64_t S1 = S0 + (lim >= kGroup ? lim / kGroup * kGroup : 0);
    if (std::max<int64_t>(N1, kSink) - S1 > R) return KVQ_ENOSPC;
    const int64_t first_in = N0 <= kSink ? kSink : kSink + (N0 - kSink + kGroup - 1) / kGroup * kGroup;
    const int64_t M = std::min(std::min(first_in, S1), N1);
    const int64_t Sj = S0 + std::max<int64_t>(0, M - S0) / kGroup * kGroup;
    const int64_t plan[8] = {N0, std::max(N0, M), S0, Sj, Sj, S1, std::max(N0, std::min(S1, N1)), N1};
    for (int i = 0; i < 8; ++i) r[i] = plan[i];
    return KVQ_OK;
}
}  // namespace

kvq_status kv_prefill_plan(int64_t n_tokens, int64_t sealed_end, int64_t n_tok, int32_t keep, int32_t ring_capacity,
                           int64_t max_ctx, int64_t ranges[8]) {
    if (!ranges || n_tok <= 0 || keep < 0 || ring_capacity <= 0 || n_tokens < 0 || sealed_end < kSink ||
        (sealed_end - kSink) % kGroup != 0)
        return KVQ_EINVAL;
    return prefill_plan(n_tokens, sealed_end, n_tok, keep, ring_capacity, max_ctx, ranges);
}

kvq_status kv_prefill(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq, int n_tok, const void* k,
                      const void* v, int keep, int64_t* groups_sealed, void* stream) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (layer < 0 || layer >= c->cfg.n_layers || n_tok <= 0 || !k || !v || !aligned16(k) || !aligned16(v) ||
        keep < c->cfg.tail)
        return KVQ_EINVAL;
    if ((st = check_seqs(c, seq_ids, n_seq)) != KVQ_OK) return st;
    // Per sequence (N0, S0 before; N1, S1 after), the plan of prefill_plan (the function the
    // test call kv_prefill_plan exposes): positions [N0, N1) split into
    //   head   [r0, r1)  the journal (and the sink): the chunk's part of groups that started
    //                    before N0, whose groups [r2, r3) are sealed from the journal right after
    //   direct [r4, r5)  groups wholly in the chunk, sealed straight from the input rows
    //   rest   [r6, r7)  the journal and, for the newest T, the exact tail
    // (r5 = S1 exceeds N1 only while the sequence is still inside the sink: S1 = 128 > N1.)
    int64_t r[kMaxSeqPerCall][8];
    for (int i = 0; i < n_seq; ++i) {
        const int s = seq_ids[i];
        const kvq_status e = prefill_plan(NT(c, layer, s), ST(c, layer, s), n_tok, keep, c->cfg.ring_capacity,
                                          c->cfg.max_ctx, r[i]);
        if (e != KVQ_OK) return e;
    }
    int64_t cnt[kMaxSeqPerCall], off[kMaxSeqPerCall], tfrom[kMaxSeqPerCall], groups[kMaxSeqPerCall];
    int64_t row[kMaxSeqPerCall];
    int64_t total = 0;
    // head, then the groups it completes (from the journal)
    for (int i = 0; i < n_seq; ++i) {
        cnt[i] = r[i][1] - r[i][0];
        off[i] = 0;
        tfrom[i] = INT64_MAX;               // older than the newest T: no tail writes
    }
    if (append_ranges(c, layer, seq_ids, n_seq, k, v, n_tok, cnt, off, tfrom, stream)) return KVQ_ECUDA;
    for (int i = 0; i < n_seq; ++i) {
        groups[i] = (r[i][3] - r[i][2]) / kGroup;
        total += groups[i];
    }
    if (seal_counts(c, layer, seq_ids, n_seq, groups, nullptr, nullptr, 0, nullptr, stream)) return KVQ_ECUDA;
    // the groups wholly in the chunk, from the input rows
    for (int i = 0; i < n_seq; ++i) {
        groups[i] = (r[i][5] - r[i][4]) / kGroup;
        row[i] = (int64_t)i * n_tok + (r[i][4] - r[i][0]);
        total += groups[i];
    }
    if (seal_counts(c, layer, seq_ids, n_seq, groups, k, v, n_tok, row, stream)) return KVQ_ECUDA;
    // the rest: the direct groups' positions count as appended (their journal slots stay unwritten)
    for (int i = 0; i < n_seq; ++i) {
        const int s = seq_ids[i];
        NT(c, layer, s) = r[i][6];
        cnt[i] = r[i][7] - r[i][6];
        off[i] = r[i][6] - r[i][0];
        tfrom[i] = r[i][7] - c->cfg.tail;
    }
    if (append_ranges(c, layer, seq_ids, n_seq, k, v, n_tok, cnt, off, tfrom, stream)) return KVQ_ECUDA;
    if (groups_sealed) *groups_sealed = total;
    return KVQ_OK;
}

kvq_status kv_seal(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq, int keep,
                   int64_t* groups_sealed, void* stream) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (layer < -1 || layer >= c->cfg.n_layers || keep < c->cfg.tail) return KVQ_EINVAL;
    if ((st = check_seqs(c, seq_ids, n_seq)) != KVQ_OK) return st;
    const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? c->cfg.n_layers : layer + 1;
    // groups per (layer, seq): every full group with S + 128 <= N - keep
    auto groups_of = [&](int l, int s) -> int64_t {
        const int64_t lim = NT(c, l, s) - keep - ST(c, l, s);
        return lim >= kGroup ? lim / kGroup : 0;
    };
    int64_t total = 0;
    int l = l0;
    while (l < l1) {
        // extend the launch over layers whose per-sequence state matches layer l
        int le = l + 1;
        auto same = [&](int a, int b) {
            for (int i = 0; i < n_seq; ++i) {
                const int s = seq_ids[i];
                if (NT(c, a, s) != NT(c, b, s) || ST(c, a, s) != ST(c, b, s)) return false;
            }
            return true;
        };
        while (le < l1 && same(l, le)) ++le;
        SealParams p{};
        p.pool = c->pool;
        p.layer0 = l;
        p.n_layers = le - l;
        p.n_seq = 0;
        int32_t acc = 0;
        for (int i = 0; i < n_seq; ++i) {
            const int s = seq_ids[i];
            const int64_t g = groups_of(l, s);
            if (g <= 0) continue;
            SealSeq& q = p.seq[p.n_seq++];
            q.slot = s;
            q.first_pos = (int32_t)ST(c, l, s);
            q.first_group = (int32_t)((ST(c, l, s) - kSink) / kGroup);
            q.n_groups = (int32_t)g;
            q.prefix = acc;
            acc += (int32_t)g;
        }
        p.groups_per_layer = acc;
        if (acc > 0) {
            if ((int64_t)acc * p.n_layers > 0x7fffffff) return KVQ_EINVAL;
            const int e = launch_seal(c->lay, p, stream);
            if (e != 0) return KVQ_ECUDA;
            for (int ll = l; ll < le; ++ll)
                for (int i = 0; i < p.n_seq; ++i)
                    ST(c, ll, p.seq[i].slot) += (int64_t)kGroup * p.seq[i].n_groups;
            total += (int64_t)acc * p.n_layers;
        }
        l = le;
    }
    if (groups_sealed) *groups_sealed = total;
    return KVQ_OK;
}

namespace {

// An integer from the environment (A/B switches of launch choices), else the default.
int getenv_int(const char* name, int dflt) {
    const char* e = std::getenv(name);
    return (e && e[0]) ? std::atoi(e) : dflt;
}

// Decode attention of one layer; with knew / vnew (the newest position's rows, fp16, already
// counted in N) the decode kernel also appends them (the fused decode step).
kvq_status decode_attn(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq, const void* q, void* out,
                       void* workspace, size_t ws_bytes, const void* knew, const void* vnew, void* stream,
                       const LaunchMarks& marks = LaunchMarks()) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (layer < 0 || layer >= c->cfg.n_layers || !q || !out || !workspace) return KVQ_EINVAL;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return KVQ_EINVAL;
    if ((st = check_seqs(c, seq_ids, n_seq)) != KVQ_OK) return st;
    const Layout& L = c->lay;
    size_t need = 0;
    kv_required_bytes(&c->cfg, nullptr, &need);
    if (ws_bytes < need) return KVQ_EINVAL;
    const size_t cap = workspace_items(c->cfg);
    AttnParams p{};
    p.pool = c->pool;
    p.q = (const uint16_t*)q;
    p.out = (uint16_t*)out;
    p.partials = (float*)workspace;
    p.knew = (const uint16_t*)knew;
    p.vnew = (const uint16_t*)vnew;
    p.layer = layer;
    p.n_seq = n_seq;
    const bool body_kernel = body_ctas_per_sm(L) > 0;
    const bool fused = body_kernel && region_kernel_ok(L);
    p.early = (marks.early && marks.pdl && fused) ? 1 : 0;
    int64_t region_tok = 0, body_groups = 0;
    for (int i = 0; i < n_seq; ++i) {
        SeqSpan& s = p.seq[i];
        s.slot = seq_ids[i];
        const int64_t N = NT(c, layer, s.slot);
        if (N <= 0) return KVQ_EINVAL;
        const int64_t S = ST(c, layer, s.slot);
        s.n_tok = (int32_t)N;
        s.body_groups = body_kernel ? (int32_t)((S - kSink) / kGroup) : 0;
        spans(L, N, S, s.lo, s.hi, s.kind, !body_kernel);
        region_tok += body_kernel ? N - (S - kSink) : N;
        body_groups += s.body_groups;
    }
    // Work items. Body items split each (sequence, head)'s groups evenly, in number proportional
    // to its groups, at most one wave of resident CTAs in all: they start first and carry most
    // of the bytes. Region items are chunks (multiples of 128 positions) of each span, about two waves'
    // worth, taken up as body items finish. (One common wave sized by estimated cost measured
    // slower: 16-bit rows cost 3 to 5 times a sealed group per position, and the minimum of one
    // item per span makes the region items too coarse.)
    const int per_sm = (L.D == 512) ? 1 : (L.D == 256 ? 2 : 4);
    const int64_t target = (int64_t)c->sm_count * per_sm;
    int64_t chunk = (region_tok * L.H + target - 1) / target;
    chunk = std::max<int64_t>(kGroup, (chunk + kGroup - 1) / kGroup * kGroup);
    int64_t body_items = (int64_t)std::max(1, fused ? decode_ctas_per_sm(L) : body_ctas_per_sm(L)) * c->sm_count;
    // at least kMinBodyGroups groups per body item where the wave would give fewer: a shorter
    // item spends most of its time on per-item set-up (query rotation, pipeline fill, partial)
    constexpr int64_t kMinBodyGroups = 6;
    body_items = std::min(body_items, std::max<int64_t>(L.H, (body_groups * L.H + kMinBodyGroups - 1) / kMinBodyGroups));
    // tq6_0 ring spans take chunks twice as long when that keeps the whole launch within one
    // wave of resident CTAs: a second, partial wave of region items costs a whole item's time
    // while most slots idle (measured on the 32k-position hybrid shape: +5.6%), whereas a launch
    // that spans several waves anyway balances better with the finer chunks
    int64_t ring_chunk = chunk;
    if (fused) {
        auto count = [&](int64_t rc) {
            int64_t n = 0;
            for (int i = 0; i < n_seq; ++i) {
                const SeqSpan& s = p.seq[i];
                for (int r = 0; r < 4; ++r) {
                    const int64_t ck = (s.kind[r] == RK_RING) ? rc : chunk;
                    n += (s.hi[r] - s.lo[r] + ck - 1) / ck;
                }
            }
            return n * L.H;
        };
        const int64_t slots = (int64_t)std::max(1, decode_ctas_per_sm(L)) * c->sm_count;
        if (body_items + count(chunk) > slots && body_items + count(2 * chunk) <= slots) ring_chunk = 2 * chunk;
    }
    // beside a tq6_0 ring, the 16-bit spans (exact tail, sink) take chunks half as long as the
    // ring's: a 16-bit position costs about twice a ring position (measured on longctx: 73 and
    // 30-42 ns per position and CTA), and a tail item of a whole ring chunk ran twice as long as
    // the ring items, ending the launch late on the SMs that drew one
    bool has_ring = false;
    for (int i = 0; i < n_seq; ++i)
        for (int r = 0; r < 4; ++r) has_ring |= p.seq[i].kind[r] == RK_RING && p.seq[i].hi[r] > p.seq[i].lo[r];
    if (has_ring) chunk = std::max<int64_t>(kGroup, ring_chunk / 2 / kGroup * kGroup);
    // without a ring, where the region items are fewer than a wave and the body items fill one,
    // the region items run in the slots the first body items to finish free (a body item's speed
    // depends on its place among the CTAs of its SM: 36 to 52 us on fa14b for equal work); 16-bit
    // spans then take 96 positions per item (two runs of the 16-bit reader at head_dim 128/256,
    // three at 512) rather than 128, which those gaps absorb better (fa14b +1.5%, its q5_1 / q4_0
    // variant +1.3%)
    if (fused && !has_ring) {
        constexpr int64_t kGapChunk = 96;
        const int64_t slots = (int64_t)std::max(1, decode_ctas_per_sm(L)) * c->sm_count;
        int64_t n_reg = 0;
        for (int i = 0; i < n_seq; ++i)
            for (int r = 0; r < 4; ++r) n_reg += (p.seq[i].hi[r] - p.seq[i].lo[r] + chunk - 1) / chunk;
        n_reg *= L.H;
        if (n_reg < slots && body_items >= slots) chunk = std::min<int64_t>(chunk, kGapChunk);
    }
    // a launch that fits in one wave of resident CTAs gives the slots left over to more, shorter
    // body items (down to kFillGroups groups each): the wave's end is set by its longest items
    if (fused) {
        constexpr int64_t kFillGroups = 4;
        const int64_t slots = (int64_t)std::max(1, decode_ctas_per_sm(L)) * c->sm_count;
        int64_t n_reg = 0;
        for (int i = 0; i < n_seq; ++i) {
            const SeqSpan& s = p.seq[i];
            for (int r = 0; r < 4; ++r) {
                const int64_t ck = (s.kind[r] == RK_RING) ? ring_chunk : chunk;
                n_reg += (s.hi[r] - s.lo[r] + ck - 1) / ck;
            }
        }
        n_reg *= L.H;
        if (body_items + n_reg < slots)
            body_items = std::max(body_items, std::min(slots - n_reg, body_groups * L.H / kFillGroups));
    }
    for (;;) {
        int64_t items = 0;
        for (int i = 0; i < n_seq; ++i) {
            SeqSpan& s = p.seq[i];
            s.items_per_head = 0;
            for (int r = 0; r < 4; ++r) {
                const int64_t ck = (s.kind[r] == RK_RING) ? ring_chunk : chunk;
                s.nchunk[r] = (int32_t)((s.hi[r] - s.lo[r] + ck - 1) / ck);
                s.items_per_head += s.nchunk[r];
            }
            s.first_item = (int32_t)items;
            items += (int64_t)s.items_per_head * L.H;
        }
        const int64_t n_region = items;
        // body items per head: largest remainders of body_items / H x groups / all groups
        const int64_t per_head = std::max<int64_t>(1, body_items / L.H);
        int64_t given = 0;
        double rem[kMaxSeqPerCall];
        for (int i = 0; i < n_seq; ++i) {
            SeqSpan& s = p.seq[i];
            s.body_per_head = 0;
            rem[i] = -1.0;
            if (s.body_groups <= 0) continue;
            const double share = (double)per_head * s.body_groups / (double)std::max<int64_t>(1, body_groups);
            s.body_per_head = (int32_t)std::max<int64_t>(1, (int64_t)share);
            rem[i] = share - (double)s.body_per_head;
            given += s.body_per_head;
        }
        while (given < per_head) {
            int best = -1;
            for (int i = 0; i < n_seq; ++i)
                if (rem[i] > -0.5 && p.seq[i].body_per_head < p.seq[i].body_groups && (best < 0 || rem[i] > rem[best]))
                    best = i;
            if (best < 0) break;
            ++p.seq[best].body_per_head;
            rem[best] = -1.0;
            ++given;
        }
        for (int i = 0; i < n_seq; ++i) {
            SeqSpan& s = p.seq[i];
            s.body_per_head = std::min(s.body_per_head, s.body_groups);
            s.body_first = (int32_t)items;
            items += (int64_t)s.body_per_head * L.H;
        }
        if ((size_t)items <= cap) {
            p.total_items = (int32_t)items;
            p.n_region_items = (int32_t)n_region;
            break;
        }
        chunk *= 2;
        ring_chunk *= 2;
        body_items = std::max<int64_t>(L.H, body_items / 2);
    }
    p.ring_chunk = (int32_t)ring_chunk;
    p.chunk = (int32_t)chunk;
    // region items at least a wave of resident CTAs (the long tq6_0 ring spans of longctx) go
    // first: launched after the body items they formed a tail of their own
    if (fused && getenv_int("KVQ_REGION_FIRST", 1)) {
        const int64_t slots = (int64_t)std::max(1, decode_ctas_per_sm(L)) * c->sm_count;
        p.region_first = p.n_region_items >= slots ? 1 : 0;
    }
    const int e = launch_decode(L, p, stream, marks);
    return e == 0 ? KVQ_OK : KVQ_ECUDA;
}

// 1 when the decode kernel of this layout can append the newest position itself: it takes the
// region items (the item that holds position N - 1 reads that row from the caller's fp16 input,
// rounded to bf16 where the row it stands for is bf16).
bool fused_append_ok(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq) {
    (void)layer; (void)seq_ids; (void)n_seq;
    const Layout& L = c->lay;
    return body_ctas_per_sm(L) > 0 && region_kernel_ok(L);
}

}  // namespace

namespace {
// The decode and merge kernels go out with programmatic stream serialization (their CTAs are
// placed while the launch ahead drains, and wait for it before touching memory), unless the
// environment sets KVQ_PDL=0.
bool pdl_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("KVQ_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}
// The decode kernel of a step's later layers reads its inputs while the previous layer's merge
// runs (AttnParams::early), unless the environment sets KVQ_EARLY=0.
bool early_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("KVQ_EARLY");
        return !(e && e[0] == '0');
    }();
    return on;
}
}  // namespace

kvq_status kv_decode_attn(kvq_cache* c, int layer, const int32_t* seq_ids, int n_seq, const void* q, void* out,
                          void* workspace, size_t ws_bytes, void* stream) {
    LaunchMarks marks;
    marks.pdl = pdl_enabled();
    return decode_attn(c, layer, seq_ids, n_seq, q, out, workspace, ws_bytes, nullptr, nullptr, stream, marks);
}

namespace {

// The launches of one decode step on `stream` (arguments checked by the caller). The caller's
// events bracket each layer's decode kernel; ev_flags: cudaEventRecordExternal while the step
// is captured into a graph (the events then become event-record nodes it can time, on a side
// branch of the graph: the kernels keep their programmatic launches), else
// cudaEventRecordDefault (the events go inline and the launches are plain).
kvq_status step_launches(kvq_cache* c, int n_layers, const int32_t* seq_ids, int n_seq, const void* q,
                         const void* k, const void* v, void* out, int seal_trigger, int keep, void* workspace,
                         size_t ws_bytes, void* const* events, int64_t* groups_sealed, void* stream,
                         unsigned ev_flags) {
    kvq_status st = KVQ_OK;
    const Layout& L = c->lay;
    const size_t qb = (size_t)n_seq * L.Hq * L.D * 2, kb = (size_t)n_seq * L.H * L.D * 2;
    int64_t total = 0;
    int32_t need[kMaxSeqPerCall];
    // Where every layer appends inside its decode kernel, the step's seals go out first, in as
    // few launches as the layers' states allow (kv_seal over all layers merges layers whose
    // lengths agree: one launch in a lockstep decode, instead of one small launch per layer
    // whose last wave leaves SMs idle). A seal reads only positions at least keep (>= T) behind
    // the newest one, so it may precede the appends; the policy decides on the lengths after them.
    bool all_fused = true;
    for (int l = 0; l < n_layers && all_fused; ++l) all_fused = fused_append_ok(c, l, seq_ids, n_seq);
    if (all_fused) {
        for (int l = 0; l < n_layers; ++l)
            for (int i = 0; i < n_seq; ++i) {
                const int s = seq_ids[i];
                const int64_t N = NT(c, l, s), S = ST(c, l, s);
                if (N + 1 > c->cfg.max_ctx) return KVQ_ENOSPC;
                if (std::max<int64_t>(N + 1, kSink) - S > c->cfg.ring_capacity) return KVQ_ENOSPC;
            }
        for (int l = 0; l < n_layers; ++l)
            for (int i = 0; i < n_seq; ++i) NT(c, l, seq_ids[i]) += 1;
        auto rollback = [&](int from) {   // the appends of layers [from, n_layers) did not go out
            for (int l = from; l < n_layers; ++l)
                for (int i = 0; i < n_seq; ++i) NT(c, l, seq_ids[i]) -= 1;
        };
        auto due = [&](int l, int32_t* out) {
            int nn = 0;
            for (int i = 0; i < n_seq; ++i) {
                const int s = seq_ids[i];
                const int64_t N = NT(c, l, s), S = ST(c, l, s);
                bool seal = false;
                if (seal_trigger > 0) seal = std::max<int64_t>(N, kSink) - S >= seal_trigger;
                else if (seal_trigger == 0) seal = N - keep - S >= kGroup;
                if (seal) out[nn++] = s;
            }
            return nn;
        };
        // the same sequences due on every layer: one call over all layers (the library merges the
        // layers whose lengths agree into one launch); otherwise one call per layer that is due
        int32_t first[kMaxSeqPerCall];
        const int n0 = due(0, first);
        bool uniform = n_layers == c->cfg.n_layers;
        for (int l = 1; l < n_layers && uniform; ++l) {
            const int nl = due(l, need);
            uniform = nl == n0 && std::equal(need, need + nl, first);
        }
        if (uniform && n0 > 0) {
            int64_t g = 0;
            st = kv_seal(c, -1, first, n0, keep, &g, stream);
            if (st != KVQ_OK) { rollback(0); return st; }
            total += g;
        } else if (!uniform) {
            for (int l = 0; l < n_layers; ++l) {
                const int nn = due(l, need);
                if (!nn) continue;
                int64_t g = 0;
                st = kv_seal(c, l, need, nn, keep, &g, stream);
                if (st != KVQ_OK) { rollback(0); return st; }
                total += g;
            }
        }
    }
    for (int l = 0; l < n_layers; ++l) {
        const char* kl = (const char*)k + l * kb;
        const char* vl = (const char*)v + l * kb;
        // the append goes into the decode kernel where it can (no separate launch); the seal,
        // when due, reads only positions at least `keep` (>= T) behind the newest one, so it
        // may run before that append
        const bool fuse = all_fused;
        if (!fuse) {
            st = kv_append(c, l, seq_ids, n_seq, 1, kl, vl, stream);
            if (st != KVQ_OK) return st;
            int nn = 0;
            for (int i = 0; i < n_seq; ++i) {
                const int s = seq_ids[i];
                const int64_t N = NT(c, l, s), S = ST(c, l, s);
                bool seal = false;
                if (seal_trigger > 0) seal = std::max<int64_t>(N, kSink) - S >= seal_trigger;
                else if (seal_trigger == 0) seal = N - keep - S >= kGroup;
                if (seal) need[nn++] = s;
            }
            if (nn) {
                int64_t g = 0;
                st = kv_seal(c, l, need, nn, keep, &g, stream);
                if (st != KVQ_OK) return st;
                total += g;
            }
        }
        LaunchMarks marks;
        const bool side = events && ev_flags == cudaEventRecordExternal;
        if (events) {
            marks.before = events[2 * l];
            marks.after = events[2 * l + 1];
            marks.flags = ev_flags;
        }
        if (!events || side) marks.pdl = pdl_enabled();
        // every layer after the first follows its predecessor's merge kernel in the stream (a
        // layer's decode launch always holds at least the newest position). Not in a pass that
        // times the decode kernels: their events would not bracket the work done early.
        marks.early = all_fused && l > 0 && !events && early_enabled();
        if (side) {
            marks.side = c->mark_stream;
            marks.fork = c->mark_fork;
        }
        st = decode_attn(c, l, seq_ids, n_seq, (const char*)q + l * qb, (char*)out + l * qb, workspace, ws_bytes,
                         fuse ? kl : nullptr, fuse ? vl : nullptr, stream, marks);
        if (st != KVQ_OK) {
            if (fuse)   // the launches that were to append the position did not go out
                for (int ll = l; ll < n_layers; ++ll)
                    for (int i = 0; i < n_seq; ++i) NT(c, ll, seq_ids[i]) -= 1;
            return st;
        }
    }
    if (events && ev_flags == cudaEventRecordExternal) {
        // join the events' side branch back into the captured stream
        if (cudaEventRecord(c->mark_fork, c->mark_stream) != cudaSuccess ||
            cudaStreamWaitEvent((cudaStream_t)stream, c->mark_fork, 0) != cudaSuccess)
            return KVQ_ECUDA;
    }
    if (groups_sealed) *groups_sealed = total;
    return KVQ_OK;
}

}  // namespace

kvq_status kv_decode_step(kvq_cache* c, int n_layers, const int32_t* seq_ids, int n_seq, const void* q,
                          const void* k, const void* v, void* out, int seal_trigger, int keep, void* workspace,
                          size_t ws_bytes, void* const* events, int64_t* groups_sealed, void* stream) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (n_layers <= 0 || n_layers > c->cfg.n_layers || !q || !k || !v || !out) return KVQ_EINVAL;
    if ((st = check_seqs(c, seq_ids, n_seq)) != KVQ_OK) return st;
    if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out) || !workspace) return KVQ_EINVAL;
    size_t ws_need = 0;
    kv_required_bytes(&c->cfg, nullptr, &ws_need);
    if (ws_bytes < ws_need) return KVQ_EINVAL;
    if (groups_sealed) *groups_sealed = 0;
    if (!c->graph_mode)
        return step_launches(c, n_layers, seq_ids, n_seq, q, k, v, out, seal_trigger, keep, workspace, ws_bytes,
                             events, groups_sealed, stream, cudaEventRecordDefault);
    // one graph per step: the host-side lengths advance while the launches are captured, and
    // go back to where they were if the step cannot be launched
    if (!c->cap_stream && cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
        return KVQ_ECUDA;
    if (events && !c->mark_stream) {
        if (cudaStreamCreateWithFlags(&c->mark_stream, cudaStreamNonBlocking) != cudaSuccess) return KVQ_ECUDA;
        if (cudaEventCreateWithFlags(&c->mark_fork, cudaEventDisableTiming) != cudaSuccess) return KVQ_ECUDA;
    }
    const std::vector<int64_t> n_tok0 = c->n_tok, sealed0 = c->sealed;
    if (cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return KVQ_ECUDA;
    int64_t g = 0;
    st = step_launches(c, n_layers, seq_ids, n_seq, q, k, v, out, seal_trigger, keep, workspace, ws_bytes, events, &g,
                       c->cap_stream, cudaEventRecordExternal);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(c->cap_stream, &graph);
    bool launched = false;
    if (st == KVQ_OK && ce == cudaSuccess && graph) {
        bool ready = false;
        if (c->step_exec) {
            cudaGraphExecUpdateResultInfo info;
            ready = cudaGraphExecUpdate(c->step_exec, graph, &info) == cudaSuccess;
            if (!ready) {
                cudaGetLastError();
                cudaGraphExecDestroy(c->step_exec);
                c->step_exec = nullptr;
            }
        }
        if (!ready) ready = cudaGraphInstantiate(&c->step_exec, graph, 0) == cudaSuccess;
        launched = ready && cudaGraphLaunch(c->step_exec, (cudaStream_t)stream) == cudaSuccess;
    }
    if (graph) cudaGraphDestroy(graph);
    if (launched) {
        if (groups_sealed) *groups_sealed = g;
        return KVQ_OK;
    }
    c->n_tok = n_tok0;
    c->sealed = sealed0;
    if (st != KVQ_OK) return st;   // an argument or capacity error: nothing was launched
    // the graph path failed: launch directly from now on
    cudaGetLastError();
    c->graph_mode = 0;
    return step_launches(c, n_layers, seq_ids, n_seq, q, k, v, out, seal_trigger, keep, workspace, ws_bytes, events,
                         groups_sealed, stream, cudaEventRecordDefault);
}

kvq_status kv_set_graph_mode(kvq_cache* c, int enable) {
    if (!c) return KVQ_EINVAL;
    c->graph_mode = enable ? 1 : 0;
    return KVQ_OK;
}

kvq_status kv_snapshot_size(const kvq_cache* c, size_t* bytes) {
    if (!c || !bytes) return KVQ_EINVAL;
    *bytes = 2 * c->n_tok.size() * sizeof(int64_t);
    return KVQ_OK;
}

kvq_status kv_snapshot(const kvq_cache* c, void* buf, size_t bytes) {
    if (!c || !buf || bytes < 2 * c->n_tok.size() * sizeof(int64_t)) return KVQ_EINVAL;
    std::memcpy(buf, c->n_tok.data(), c->n_tok.size() * sizeof(int64_t));
    std::memcpy((char*)buf + c->n_tok.size() * sizeof(int64_t), c->sealed.data(), c->sealed.size() * sizeof(int64_t));
    return KVQ_OK;
}

kvq_status kv_restore(kvq_cache* c, const void* buf, size_t bytes) {
    if (!c || !buf || bytes < 2 * c->n_tok.size() * sizeof(int64_t)) return KVQ_EINVAL;
    std::memcpy(c->n_tok.data(), buf, c->n_tok.size() * sizeof(int64_t));
    std::memcpy(c->sealed.data(), (const char*)buf + c->n_tok.size() * sizeof(int64_t), c->sealed.size() * sizeof(int64_t));
    return KVQ_OK;
}

kvq_status kv_state(const kvq_cache* c, int layer, int seq, int64_t* n_tokens, int64_t* sealed_end) {
    if (!c || layer < 0 || layer >= c->cfg.n_layers || seq < 0 || seq >= c->cfg.max_seqs) return KVQ_EINVAL;
    const size_t i = (size_t)layer * c->cfg.max_seqs + seq;
    if (n_tokens) *n_tokens = c->n_tok[i];
    if (sealed_end) *sealed_end = c->sealed[i];
    return KVQ_OK;
}

kvq_status kv_get_status(kvq_cache* c, uint32_t* word) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    uint32_t w = 0;
    if (cudaMemcpy(&w, (char*)c->pool + c->lay.status_off, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ECUDA;
    if (w && cudaMemset((char*)c->pool + c->lay.status_off, 0, 4) != cudaSuccess) return KVQ_ECUDA;
    if (word) *word = w;
    return w ? KVQ_EDEVICE : KVQ_OK;
}

kvq_status kv_test_wait_timeout(kvq_cache* c, uint64_t limit_ns, void* stream) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (limit_ns < 1000 || limit_ns > 10000000000ull) return KVQ_EINVAL;
    return launch_wait_probe(c->lay, c->pool, limit_ns, stream) == 0 ? KVQ_OK : KVQ_ECUDA;
}

kvq_status kv_dequant(kvq_cache* c, int layer, int seq, int head, int which, int64_t p0, int64_t n, float* out,
                      void* stream) {
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (layer < 0 || layer >= c->cfg.n_layers || seq < 0 || seq >= c->cfg.max_seqs || head < 0 ||
        head >= c->cfg.n_kv_heads || (which != 0 && which != 1) || !out || p0 < 0 || n <= 0)
        return KVQ_EINVAL;
    const int64_t N = NT(c, layer, seq), S = ST(c, layer, seq);
    if (p0 + n > N) return KVQ_EINVAL;
    int32_t lo[4], hi[4], kind[4];
    const int ns = spans(c->lay, N, S, lo, hi, kind, true);
    for (int r = 0; r < ns; ++r) {
        const int64_t a = std::max<int64_t>(lo[r], p0), b = std::min<int64_t>(hi[r], p0 + n);
        if (b <= a) continue;
        const int e = launch_dequant(c->lay, c->pool, layer, seq, head, which, kind[r], a, b - a,
                                     out + (a - p0) * c->lay.D, stream);
        if (e != 0) return KVQ_ECUDA;
    }
    return KVQ_OK;
}

kvq_status kv_region_ptr(const kvq_cache* c, int layer, int seq, int head, int which, int region, void** ptr,
                         size_t* bytes) {
    if (!c || !ptr || layer < 0 || layer >= c->cfg.n_layers || seq < 0 || seq >= c->cfg.max_seqs || head < 0 ||
        head >= c->cfg.n_kv_heads || (which != 0 && which != 1))
        return KVQ_EINVAL;
    const Layout& L = c->lay;
    const int64_t u = L.unit(layer, seq, head);
    int64_t off = 0, sz = 0;
    const bool tq = L.journal == KVQ_TQ6_0;
    switch (region) {
        case KVQ_REGION_SINK: off = L.sink_off[which] + u * L.sink_stride[which]; sz = (int64_t)kSink * L.D * 2; break;
        case KVQ_REGION_JOURNAL: off = L.jcode_off[which] + u * L.jcode_stride[which]; sz = (int64_t)L.R * L.jrow_bytes; break;
        case KVQ_REGION_JOURNAL_SCALE:
            if (!tq) return KVQ_EINVAL;
            off = L.jscale_off[which] + u * L.jscale_stride[which]; sz = (int64_t)L.R * (L.D / 128) * 2; break;
        case KVQ_REGION_TAIL:
            if (!tq) return KVQ_EINVAL;
            off = L.tail_off[which] + u * L.tail_stride[which]; sz = (int64_t)L.T * L.D * 2; break;
        case KVQ_REGION_BODY: off = L.body_off[which] + u * L.body_stride[which]; sz = (int64_t)L.gcap * L.rec_bytes[which]; break;
        default: return KVQ_EINVAL;
    }
    *ptr = (char*)c->pool + off;
    if (bytes) *bytes = (size_t)sz;
    return KVQ_OK;
}

kvq_status kv_format_tables(float centroids[16], float boundaries[15], uint64_t sign_words[4]) {
    const FormatTables& t = host_tables();
    if (centroids) std::memcpy(centroids, t.cent, sizeof(t.cent));
    if (boundaries) std::memcpy(boundaries, t.bnd, sizeof(t.bnd));
    if (sign_words) std::memcpy(sign_words, t.sign_words, sizeof(t.sign_words));
    return KVQ_OK;
}

kvq_status kv_format_tables_turbo3(float centroids[8], float boundaries[7]) {
    const FormatTables& t = host_tables();
    if (centroids) std::memcpy(centroids, t.cent3, sizeof(t.cent3));
    if (boundaries) std::memcpy(boundaries, t.bnd3, sizeof(t.bnd3));
    return KVQ_OK;
}

}  // extern "C"
