// Host side of the C ABI declared in waste_moe.h: argument and record checks,
// workspace, statistics, error strings, and the launch sequence of each call.
#include "common.cuh"
#include "lut_dev.cuh"

#include <algorithm>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

using namespace wm;

struct waste_moe {
    waste_moe_config cfg;
    LayerView L;
    Workspace W;
    int num_sms;
    int lookahead;
    int max_slots;
    int pred_P; // experts per token of the last prefetch into this layer
    bool profiling;
    Timing route_tm, fwd_tm, step_tm;
    unsigned long long *trace; // caller's trace buffer for the step kernel, or null
    int trace_cap;
    int mma_min_tokens; // tokens an expert needs in one call to take the tensor-core path
    waste_bank *bank;   // records live in this bank (layer bank_layer), or null
    int bank_layer;
    // the lookahead inside the step (waste_moe_set_lookahead): the next layer and P, and whether
    // the last route also ran the next layer's router rows (the forward then predicts)
    waste_moe *ahead_next;
    int ahead_P;
    bool ahead_routed;
};

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int ok() {
    g_err.clear();
    return WASTE_OK;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(WASTE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_config(const waste_moe_config *c) {
    if (!c) return fail(WASTE_EINVAL, "config is NULL");
    if (c->abi_version != WASTE_MOE_ABI_VERSION)
        return fail(WASTE_EINVAL, "abi_version %u, library speaks %u", c->abi_version, WASTE_MOE_ABI_VERSION);
    if (c->d <= 0 || c->d % kVec) return fail(WASTE_EINVAL, "d = %d must be a positive multiple of 8", c->d);
    if (c->f <= 0 || c->f % kVec) return fail(WASTE_EINVAL, "f = %d must be a positive multiple of 8", c->f);
    if (c->n_experts < 1 || c->n_experts > kMaxExperts)
        return fail(WASTE_EINVAL, "n_experts = %d outside [1, %d]", c->n_experts, kMaxExperts);
    if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > kMaxTopK)
        return fail(WASTE_EINVAL, "top_k = %d outside [1, min(n_experts, %d)]", c->top_k, kMaxTopK);
    if (c->act_dtype != WASTE_ACT_F32 && c->act_dtype != WASTE_ACT_BF16)
        return fail(WASTE_EINVAL, "act_dtype = %d", c->act_dtype);
    if (c->max_tokens < 1) return fail(WASTE_EINVAL, "max_tokens = %d", c->max_tokens);
    if (c->lookahead < 0 || c->lookahead > kMaxTopK || c->lookahead > c->n_experts)
        return fail(WASTE_EINVAL, "lookahead = %d outside [0, min(n_experts, %d)]", c->lookahead, kMaxTopK);
    const uint32_t known = WASTE_FLAG_VERIFY_CRC | WASTE_FLAG_FORCE_GEMV | WASTE_FLAG_FORCE_MMA |
                           WASTE_FLAG_K2_RECONSTRUCT | WASTE_FLAG_STEP_KERNEL | WASTE_FLAG_BANK_SERIAL;
    if (c->flags & ~known) return fail(WASTE_EINVAL, "unknown flags 0x%x", c->flags & ~known);
    return WASTE_OK;
}

void layout(const waste_moe_config *c, size_t *stride, size_t off[3], size_t bytes[3]) {
    const MatGeom gu = mat_geom(c->f, c->d), dn = mat_geom(c->d, c->f);
    bytes[0] = bytes[1] = round_up(gu.chunk_bytes(), WASTE_RECORD_ALIGN);
    bytes[2] = round_up(dn.chunk_bytes(), WASTE_RECORD_ALIGN);
    off[0] = WASTE_RECORD_ALIGN;
    off[1] = off[0] + bytes[0];
    off[2] = off[1] + bytes[1];
    *stride = off[2] + bytes[2];
}

} // namespace

namespace wm {
void set_last_error(const char *msg) { g_err = msg; }

// One CTA running the bounded wait that the step kernel's work items use between one
// another, on a caller-owned counter.
__global__ void __launch_bounds__(32) debug_wait_kernel(const unsigned *c, unsigned target, uint32_t *err,
                                                        unsigned long long limit_ns) {
    lut::wait_counter(c, target, err, limit_ns);
}

int device_sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}
} // namespace wm

extern "C" {

const char *waste_moe_last_error(void) { return g_err.c_str(); }

int waste_moe_record_layout(const waste_moe_config *cfg, size_t *record_stride,
                            size_t section_offset[3], size_t section_bytes[3]) {
    int rc = check_config(cfg);
    if (rc) return rc;
    size_t st, off[3], by[3];
    layout(cfg, &st, off, by);
    if (record_stride) *record_stride = st;
    for (int m = 0; m < 3; ++m) {
        if (section_offset) section_offset[m] = off[m];
        if (section_bytes) section_bytes[m] = by[m];
    }
    return ok();
}

int waste_moe_pack_records(const waste_moe_config *cfg, int32_t layer, int32_t expert_begin,
                           int32_t n_experts, const uint8_t *d_gate_codes,
                           const uint8_t *d_up_codes, const uint8_t *d_down_codes,
                           uint8_t *d_records, size_t record_stride, int32_t compute_crc,
                           waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    int rc = check_config(cfg);
    if (rc) return rc;
    if (n_experts < 0 || expert_begin < 0 || expert_begin + n_experts > cfg->n_experts)
        return fail(WASTE_EINVAL, "experts [%d, %d) outside [0, %d)", expert_begin,
                    expert_begin + n_experts, cfg->n_experts);
    if (n_experts == 0) return ok();
    if (!d_gate_codes || !d_up_codes || !d_down_codes || !d_records)
        return fail(WASTE_EINVAL, "NULL code or record pointer");
    if (!aligned(d_records, WASTE_RECORD_ALIGN))
        return fail(WASTE_ELAYOUT, "record bank base %p is not 4096-aligned", (const void *)d_records);
    size_t st, off[3], by[3];
    layout(cfg, &st, off, by);
    if (record_stride < st || record_stride % WASTE_RECORD_ALIGN)
        return fail(WASTE_ELAYOUT, "record stride %zu: needs a multiple of 4096 >= %zu", record_stride, st);
    waste_record_header hdr;
    memset(&hdr, 0, sizeof hdr);
    hdr.magic = WASTE_RECORD_MAGIC;
    hdr.version = WASTE_RECORD_VERSION;
    hdr.layer = layer;
    hdr.d = cfg->d;
    hdr.f = cfg->f;
    hdr.n_stages = kStages;
    hdr.codebook_size = kCodes;
    hdr.vec = kVec;
    hdr.layout_id = WASTE_LAYOUT_TILED16X;
    for (int m = 0; m < 3; ++m) {
        hdr.section_offset[m] = off[m];
        hdr.section_bytes[m] = by[m];
    }
    hdr.record_bytes = record_stride;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *first = d_records + (size_t)expert_begin * record_stride;
    cudaError_t e = launch_headers(first, record_stride, n_experts, hdr, expert_begin, s);
    if (e != cudaSuccess) return cuda_fail(e, "header kernel");
    e = launch_pack(mat_geom(cfg->f, cfg->d), mat_geom(cfg->d, cfg->f), n_experts, d_gate_codes,
                    d_up_codes, d_down_codes, first, record_stride, off, s);
    if (e != cudaSuccess) return cuda_fail(e, "pack kernel");
    if (compute_crc) {
        // payload crc32 into each header: a temporary device buffer, then a wait on the stream
        const size_t payload = by[0] + by[1] + by[2];
        uint32_t *scratch = nullptr;
        const size_t words = crc_scratch_words(payload, n_experts);
        e = cudaMalloc(&scratch, words * 4);
        if (e != cudaSuccess) return cuda_fail(e, "crc scratch");
        uint32_t *crc = scratch + (words - (size_t)n_experts);
        e = launch_payload_crc(first, record_stride, n_experts, off[0], payload, scratch, crc, device_sm_count(), s);
        if (e == cudaSuccess)
            e = launch_crc_store(crc, first, record_stride, n_experts, offsetof(waste_record_header, payload_crc32),
                                 s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        cudaFree(scratch);
        if (e != cudaSuccess) return cuda_fail(e, "payload crc32");
    }
    return ok();
}

int waste_moe_create(const waste_moe_config *cfg, const float *d_router_w,
                     const float *d_router_bias, const uint8_t *d_records, size_t record_stride,
                     const float *d_codebooks, waste_moe **out) {
    const NvtxRange nvtx_range(__func__);
    if (!out) return fail(WASTE_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = check_config(cfg);
    if (rc) return rc;
    if (!d_router_w || !d_records || !d_codebooks)
        return fail(WASTE_EINVAL, "NULL router, record or codebook pointer");
    if (!aligned(d_router_w, 16) || !aligned(d_codebooks, 16) ||
        (d_router_bias && !aligned(d_router_bias, 4)))
        return fail(WASTE_EINVAL, "router / codebook pointers must be 16-byte aligned");
    if (!aligned(d_records, WASTE_RECORD_ALIGN))
        return fail(WASTE_ELAYOUT, "record bank base %p is not 4096-aligned", (const void *)d_records);
    size_t st, off[3], by[3];
    layout(cfg, &st, off, by);
    if (record_stride < st || record_stride % WASTE_RECORD_ALIGN)
        return fail(WASTE_ELAYOUT, "record stride %zu: needs a multiple of 4096 >= %zu", record_stride, st);

    // ---- record headers: one strided copy, then every field checked
    const int E = cfg->n_experts;
    std::vector<waste_record_header> hdrs((size_t)E);
    cudaError_t ce = cudaMemcpy2D(hdrs.data(), sizeof(waste_record_header), d_records, record_stride,
                                  sizeof(waste_record_header), (size_t)E, cudaMemcpyDefault);
    if (ce != cudaSuccess) return cuda_fail(ce, "copying record headers");
    for (int e = 0; e < E; ++e) {
        const waste_record_header &h = hdrs[(size_t)e];
        if (h.magic != WASTE_RECORD_MAGIC)
            return fail(WASTE_ELAYOUT, "record %d: bad magic 0x%08x", e, h.magic);
        if (h.version != WASTE_RECORD_VERSION)
            return fail(WASTE_ELAYOUT, "record %d: version %u", e, h.version);
        if (h.expert_id != e) return fail(WASTE_ELAYOUT, "record %d holds expert id %d", e, h.expert_id);
        if (cfg->layer >= 0 && h.layer != cfg->layer)
            return fail(WASTE_ELAYOUT, "record %d: layer %d, expected %d", e, h.layer, cfg->layer);
        if (h.d != cfg->d || h.f != cfg->f || h.n_stages != kStages || h.codebook_size != kCodes ||
            h.vec != kVec)
            return fail(WASTE_ELAYOUT, "record %d: shapes (d %d, f %d, %d x %d x %d) do not match", e, h.d,
                        h.f, h.n_stages, h.codebook_size, h.vec);
        if (h.layout_id != WASTE_LAYOUT_TILED16X)
            return fail(WASTE_ELAYOUT, "record %d: unknown code layout %u", e, h.layout_id);
        for (int m = 0; m < 3; ++m) {
            if (h.section_offset[m] % WASTE_RECORD_ALIGN || h.section_offset[m] < WASTE_RECORD_ALIGN ||
                h.section_bytes[m] < by[m] || h.section_offset[m] + h.section_bytes[m] > record_stride ||
                h.section_offset[m] != off[m])
                return fail(WASTE_ELAYOUT, "record %d: section %d at %llu (+%llu) outside the record", e, m,
                            (unsigned long long)h.section_offset[m], (unsigned long long)h.section_bytes[m]);
        }
    }

    // ---- payload crc32 of every record against its header (WASTE_FLAG_VERIFY_CRC)
    if (cfg->flags & WASTE_FLAG_VERIFY_CRC) {
        for (int e = 0; e < E; ++e)
            if (hdrs[(size_t)e].payload_crc32 == 0)
                return fail(WASTE_ECRC, "record %d carries no payload crc32 (packed without one)", e);
        const size_t payload = by[0] + by[1] + by[2];
        const size_t words = crc_scratch_words(payload, E);
        uint32_t *scratch = nullptr;
        ce = cudaMalloc(&scratch, words * 4);
        if (ce != cudaSuccess) {
            cudaGetLastError();
            return fail(WASTE_ENOMEM, "crc scratch of %zu bytes", words * 4);
        }
        uint32_t *crc = scratch + (words - (size_t)E);
        std::vector<uint32_t> got((size_t)E);
        ce = launch_payload_crc(d_records, record_stride, E, off[0], payload, scratch, crc, device_sm_count(), 0);
        if (ce == cudaSuccess) ce = cudaMemcpy(got.data(), crc, (size_t)E * 4, cudaMemcpyDeviceToHost);
        cudaFree(scratch);
        if (ce != cudaSuccess) return cuda_fail(ce, "payload crc32");
        for (int e = 0; e < E; ++e)
            if (got[(size_t)e] != hdrs[(size_t)e].payload_crc32)
                return fail(WASTE_ECRC, "record %d: payload crc32 0x%08x, header says 0x%08x", e, got[(size_t)e],
                            hdrs[(size_t)e].payload_crc32);
    }

    waste_moe *H = new (std::nothrow) waste_moe();
    if (!H) return fail(WASTE_ENOMEM, "host allocation");
    H->cfg = *cfg;
    H->num_sms = device_sm_count();
    H->lookahead = cfg->lookahead;
    if (const char *env = getenv("WASTE_LOOKAHEAD")) {
        const int v = atoi(env);
        if (v >= 0 && v <= kMaxTopK && v <= E) H->lookahead = v;
    }
    H->max_slots = cfg->max_tokens * cfg->top_k;
    H->pred_P = 0;
    H->profiling = false;
    H->trace = nullptr;
    H->trace_cap = 0;
    H->bank = nullptr;
    H->bank_layer = 0;
    H->ahead_next = nullptr;
    H->ahead_P = 0;
    H->ahead_routed = false;
    LayerView &L = H->L;
    L.router_w = d_router_w;
    L.router_b = d_router_bias;
    L.records = d_records;
    L.slot_map = nullptr;
    L.stride = record_stride;
    for (int m = 0; m < 3; ++m) L.sec_off[m] = off[m];
    L.codebooks = d_codebooks;
    L.d = cfg->d;
    L.f = cfg->f;
    L.E = E;
    L.k = cfg->top_k;
    L.act_bf16 = cfg->act_dtype == WASTE_ACT_BF16;
    L.gu = mat_geom(cfg->f, cfg->d);
    L.dn = mat_geom(cfg->d, cfg->f);

    H->mma_min_tokens = kDefaultMmaMinTokens;
    if (const char *env = getenv("WASTE_MMA_MIN_TOKENS")) {
        const int v = atoi(env);
        if (v >= 1) H->mma_min_tokens = v;
    }
    if (cfg->flags & WASTE_FLAG_FORCE_MMA) H->mma_min_tokens = 1;

    // ---- workspace, one allocation carved into 256-byte aligned pieces
    const size_t T = (size_t)cfg->max_tokens, S = (size_t)H->max_slots;
    const size_t npair = (size_t)(L.dn.nseg + 1) / 2;
    // grouping of batched calls (any call with more than one token, or every call
    // under WASTE_FLAG_FORCE_MMA)
    const bool grouped = cfg->max_tokens > 1 || (cfg->flags & WASTE_FLAG_FORCE_MMA);
    const size_t max_chunks = (size_t)E + S / kGroupTokens + 1;
    const size_t G = grouped ? 1 : 0;
    size_t sizes[] = {
        T * E * 4,                                  // logits
        T * E * 4,                                  // logits_lo
        T * E * 4,                                  // pred_logits
        T * kMaxTopK * 4,                           // pred_idx
        T * 4,                                      // pred_count
        T * kMaxTopK * 4,                           // pred_gate_sel
        S * (size_t)((L.gu.nseg + 1) / 2) * 2 * (size_t)L.f * 4, // part_gu
        S * npair * (size_t)L.d * 4,                // part_dn
        kStatCount * 8,                             // stats
        4,                                          // err
        (4 + 2 * S + kMaxFusedRowBlocks) * 4,       // sync
        S * 4,                                      // bank_wait
        S * 4,                                      // bank_order
        4,                                          // route_done
        G * ((size_t)E + 1) * 4,                    // grp.offs
        G * S * 4,                                  // grp.sorted
        G * S * 4,                                  // grp.lut_slots
        G * max_chunks * 16,                        // grp.chunks
        G * 2 * 4,                                  // grp.counts
        G * S,                                      // grp.one_part
        G * grouped_tile_rows((int)S, (int)max_chunks) * ((L.d + 63) / 64) * 128, // grp.xg
        G * grouped_tile_rows((int)S, (int)max_chunks) * ((L.f + 63) / 64) * 128, // grp.ag
        (T > 16 ? (size_t)kRouterMaxSplits * T * E * 4 : 0), // router_part
        (size_t)E * 8,                              // route_slots
        (size_t)E * 8,                              // ahead_keys
    };
    const int n_parts = (int)(sizeof sizes / sizeof sizes[0]);
    size_t offs[32], total = 0;
    for (int i = 0; i < n_parts; ++i) {
        offs[i] = total;
        total += round_up(sizes[i], 256);
    }
    void *base = nullptr;
    ce = cudaMalloc(&base, total);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        delete H;
        return fail(WASTE_ENOMEM, "workspace of %zu bytes: %s", total, cudaGetErrorString(ce));
    }
    char *b = static_cast<char *>(base);
    Workspace &W = H->W;
    W.base = base;
    W.bytes = total;
    W.logits = reinterpret_cast<float *>(b + offs[0]);
    W.logits_lo = reinterpret_cast<float *>(b + offs[1]);
    W.pred_logits = reinterpret_cast<float *>(b + offs[2]);
    W.pred_idx = reinterpret_cast<int32_t *>(b + offs[3]);
    W.pred_count = reinterpret_cast<int32_t *>(b + offs[4]);
    W.pred_gate_sel = reinterpret_cast<float *>(b + offs[5]);
    W.pred_idx_sel = W.pred_idx;
    W.part_gu = reinterpret_cast<float *>(b + offs[6]);
    W.part_dn = reinterpret_cast<float *>(b + offs[7]);
    W.stats = reinterpret_cast<unsigned long long *>(b + offs[8]);
    W.err = reinterpret_cast<uint32_t *>(b + offs[9]);
    W.sync = reinterpret_cast<unsigned *>(b + offs[10]);
    W.bank_wait = reinterpret_cast<int32_t *>(b + offs[11]);
    W.bank_order = reinterpret_cast<int32_t *>(b + offs[12]);
    W.route_done = reinterpret_cast<unsigned *>(b + offs[13]);
    Grouping &Gp = W.grp;
    Gp.offs = grouped ? reinterpret_cast<int32_t *>(b + offs[14]) : nullptr;
    Gp.sorted = grouped ? reinterpret_cast<int32_t *>(b + offs[15]) : nullptr;
    Gp.lut_slots = grouped ? reinterpret_cast<int32_t *>(b + offs[16]) : nullptr;
    Gp.chunks = grouped ? reinterpret_cast<int4 *>(b + offs[17]) : nullptr;
    Gp.counts = grouped ? reinterpret_cast<int32_t *>(b + offs[18]) : nullptr;
    Gp.one_part = grouped ? reinterpret_cast<uint8_t *>(b + offs[19]) : nullptr;
    Gp.xg = grouped ? reinterpret_cast<uint8_t *>(b + offs[20]) : nullptr;
    Gp.ag = grouped ? reinterpret_cast<uint8_t *>(b + offs[21]) : nullptr;
    Gp.max_chunks = grouped ? (int)max_chunks : 0;
    W.router_part = T > 16 ? reinterpret_cast<float *>(b + offs[22]) : nullptr;
    W.ahead_keys = reinterpret_cast<unsigned long long *>(b + offs[24]);
    W.route_slots = reinterpret_cast<unsigned long long *>(b + offs[23]);
    ce = cudaMemset(base, 0, total);
    if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
    if (ce != cudaSuccess) {
        cudaFree(base);
        delete H;
        return cuda_fail(ce, "clearing the workspace");
    }
    *out = H;
    return ok();
}

static void drop_events(waste_moe *h) {
    if (!h->profiling) return;
    for (int i = 0; i < 8; ++i) {
        cudaEventDestroy(h->route_tm.ev[i]);
        cudaEventDestroy(h->fwd_tm.ev[i]);
        cudaEventDestroy(h->step_tm.ev[i]);
    }
    h->profiling = false;
}

void waste_moe_destroy(waste_moe *h) {
    if (!h) return;
    cudaDeviceSynchronize();
    drop_events(h);
    cudaFree(h->W.base);
    delete h;
}

int waste_moe_set_profiling(waste_moe *h, int32_t enable) {
    if (!h) return fail(WASTE_EINVAL, "NULL handle");
    if (!enable) {
        cudaDeviceSynchronize();
        drop_events(h);
        return ok();
    }
    if (h->profiling) return ok();
    for (int i = 0; i < 8; ++i) {
        cudaError_t e = cudaEventCreate(&h->route_tm.ev[i]);
        if (e == cudaSuccess) e = cudaEventCreate(&h->fwd_tm.ev[i]);
        if (e == cudaSuccess) e = cudaEventCreate(&h->step_tm.ev[i]);
        if (e != cudaSuccess) return cuda_fail(e, "creating profiling events");
    }
    h->route_tm.n = h->fwd_tm.n = h->step_tm.n = 0;
    h->profiling = true;
    return ok();
}

int waste_moe_read_profile(const waste_moe *h, float ms[6]) {
    if (!h || !ms) return fail(WASTE_EINVAL, "NULL handle or output");
    if (!h->profiling) return fail(WASTE_EINVAL, "profiling is not enabled");
    for (int i = 0; i < 6; ++i) ms[i] = -1.f;
    const Timing *t[3] = {&h->route_tm, &h->fwd_tm, &h->step_tm};
    const int count[3] = {3, 4, 2};
    int o = 0;
    for (int j = 0; j < 3; ++j) {
        const int n = count[j];
        // the forward with its gate/up and down units in one launch records 3 events:
        // that launch into ms[2], the combine into ms[4], ms[3] stays -1; a route whose
        // router took the top-k records 2 (ms[1] stays -1)
        const bool one_launch = j == 1 && t[j]->n == 3;
        if (t[j]->n == n || one_launch || (j == 0 && t[j]->n == 2)) {
            const int m = t[j]->n;
            cudaError_t e = cudaEventSynchronize(t[j]->ev[m - 1]);
            if (e != cudaSuccess) return cuda_fail(e, "waiting for profiling events");
            for (int i = 0; i + 1 < m; ++i) {
                const int at = one_launch && i == 1 ? o + 2 : o + i;
                e = cudaEventElapsedTime(&ms[at], t[j]->ev[i], t[j]->ev[i + 1]);
                if (e != cudaSuccess) return cuda_fail(e, "reading profiling events");
            }
        }
        o += n - 1;
    }
    return ok();
}

static int check_tokens(const waste_moe *h, int32_t T, const void *d_h) {
    if (!h) return fail(WASTE_EINVAL, "handle is NULL");
    if (T < 0 || T > h->cfg.max_tokens)
        return fail(WASTE_EINVAL, "T = %d outside [0, max_tokens = %d]", T, h->cfg.max_tokens);
    if (T > 0 && !d_h) return fail(WASTE_EINVAL, "hidden states pointer is NULL");
    if (d_h && !aligned(d_h, 16)) return fail(WASTE_EINVAL, "hidden states must be 16-byte aligned");
    return WASTE_OK;
}

int waste_moe_route(waste_moe *h, const void *d_h, int32_t T, int32_t *d_idx, float *d_gate,
                    float *d_logits, waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    int rc = check_tokens(h, T, d_h);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!d_idx || !d_gate) return fail(WASTE_EINVAL, "NULL idx or gate output");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float *logits = d_logits ? d_logits : h->W.logits;
    if (h->profiling) cudaEventRecord(h->route_tm.ev[0], s);
    const unsigned long long router_bytes = (unsigned long long)h->L.E * (unsigned long long)h->L.d * 4ull;
    const int pred_stride = h->pred_P > 0 ? h->pred_P : 1;
    RouteTopk F{h->W.route_done, h->L.k, d_idx, d_gate, h->W.pred_idx, h->W.pred_count, pred_stride, h->W.stats,
                router_bytes, h->W.route_slots};
    // the lookahead inside the step: the next layer's router rows ride on this launch
    const waste_moe *nx = h->ahead_next;
    h->ahead_routed = false;
    if (nx && h->ahead_P > 0 && T == 1 && nx->L.d == h->L.d && nx->L.act_bf16 == h->L.act_bf16 &&
        ((uintptr_t)nx->L.router_w & 15) == 0 && route_polled_fits(h->L, d_h, T, nx->L.E, h->num_sms)) {
        F.ahead_w = nx->L.router_w;
        F.ahead_b = nx->L.router_b;
        F.ahead_E = nx->L.E;
        F.ahead_keys = nx->W.ahead_keys;
        h->ahead_routed = true;
    }
    bool fused = false;
    cudaError_t e = launch_router(h->L, d_h, T, logits, h->W.logits_lo, s, h->W.router_part, h->num_sms, &F, &fused,
                                  h->W.err);
    if (e != cudaSuccess) return cuda_fail(e, "router kernel");
    if (h->profiling) cudaEventRecord(h->route_tm.ev[1], s);
    if (!fused) {
        e = launch_topk(logits, h->W.logits_lo, T, h->L.E, h->L.k, d_idx, d_gate, h->W.pred_idx,
                        h->W.pred_count, pred_stride, h->W.stats, router_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "top-k kernel");
    }
    if (h->profiling) {
        if (fused) {
            h->route_tm.n = 2; // the router's last CTA took the top-k: no top-k kernel
        } else {
            cudaEventRecord(h->route_tm.ev[2], s);
            h->route_tm.n = 3;
        }
    }
    return ok();
}

// Grouped tensor-core path: bf16 activations and more than one token, or every call
// under WASTE_FLAG_FORCE_MMA; never under WASTE_FLAG_FORCE_GEMV.
static bool use_grouped(const waste_moe *h, int T) {
    if (!h->W.grp.xg || (h->cfg.flags & WASTE_FLAG_FORCE_GEMV)) return false;
    if (h->cfg.flags & WASTE_FLAG_FORCE_MMA) return true;
    return h->cfg.act_dtype == WASTE_ACT_BF16 && T > 1;
}

int waste_moe_forward(waste_moe *h, const void *d_h, int32_t T, const int32_t *d_idx,
                      const float *d_gate, float *d_out, int32_t mode, waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    int rc = check_tokens(h, T, d_h);
    if (rc) return rc;
    if (mode < 0 || mode > 2) return fail(WASTE_EINVAL, "mode = %d", mode);
    if (mode == 2 && h->cfg.act_dtype != WASTE_ACT_F32)
        return fail(WASTE_EINVAL, "mode 2 (out = h + y) needs fp32 hidden states");
    // whether the route in front of this call ran the next layer's router rows (consumed here)
    const bool ahead = h->ahead_routed;
    h->ahead_routed = false;
    if (T == 0) return ok();
    if (!d_idx || !d_gate || !d_out) return fail(WASTE_EINVAL, "NULL idx, gate or out");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool recon = (h->cfg.flags & WASTE_FLAG_K2_RECONSTRUCT) != 0;
    cudaError_t e;
    if (h->bank && !(h->cfg.flags & WASTE_FLAG_BANK_SERIAL) && !use_grouped(h, T) &&
        T * h->L.k <= kOverlapMaxSlots && fused_eligible(h->L, T, false, h->num_sms)) {
        // the routed experts' copy runs inside the step kernel, each expert consumed on arrival
        BankLanes lanes;
        e = launch_bank_plan_overlap(h->bank, h->bank_layer, d_idx, T * h->L.k, h->W.bank_wait, h->W.bank_order,
                                     &lanes, s);
        if (e != cudaSuccess) return cuda_fail(e, "bank plan");
        if (h->profiling) cudaEventRecord(h->step_tm.ev[0], s);
        e = launch_fused_step(h->L, h->W, d_h, T, false, const_cast<int32_t *>(d_idx),
                              const_cast<float *>(d_gate), nullptr, nullptr, nullptr, 1, d_out, mode,
                              recon, h->num_sms, s, h->trace, h->trace_cap, &lanes, h->W.bank_order);
        if (h->profiling) {
            cudaEventRecord(h->step_tm.ev[1], s);
            h->step_tm.n = 2;
            h->fwd_tm.n = 0;
        }
        if (e != cudaSuccess) return cuda_fail(e, "banked step kernel");
        return ok();
    }
    if (h->bank) {
        // the routed experts into the bank's HBM cache before the expert kernels read them
        e = launch_bank_fetch(h->bank, h->bank_layer, d_idx, T * h->L.k, true, s);
        if (e != cudaSuccess) return cuda_fail(e, "bank fetch");
    }
    if (use_grouped(h, T)) {
        e = launch_grouped_forward(h->L, h->W, d_h, T, d_idx, d_gate, d_out, mode, h->mma_min_tokens, recon,
                                   h->num_sms, s, h->profiling ? &h->fwd_tm : nullptr);
        if (h->profiling) h->step_tm.n = 0;
    } else if ((h->cfg.flags & WASTE_FLAG_STEP_KERNEL) && !h->bank && fused_eligible(h->L, T, false, h->num_sms)) {
        if (h->profiling) cudaEventRecord(h->step_tm.ev[0], s);
        e = launch_fused_step(h->L, h->W, d_h, T, false, const_cast<int32_t *>(d_idx),
                              const_cast<float *>(d_gate), nullptr, nullptr, nullptr, 1, d_out, mode,
                              recon, h->num_sms, s, h->trace, h->trace_cap);
        if (h->profiling) {
            cudaEventRecord(h->step_tm.ev[1], s);
            h->step_tm.n = 2;
            h->fwd_tm.n = 0;
        }
    } else {
        // the lookahead inside the step, when the route that produced d_idx also ran the next
        // layer's router rows
        LutAhead LA{};
        if (ahead && h->ahead_next && T == 1) {
            waste_moe *nx = h->ahead_next;
            LA.keys = nx->W.ahead_keys;
            LA.E = nx->L.E;
            LA.P = h->ahead_P;
            LA.pred_idx = nx->W.pred_idx;
            LA.pred_count = nx->W.pred_count;
            LA.records = nx->L.records;
            LA.stride = nx->L.stride;
            LA.off_gate = nx->L.sec_off[0];
            LA.off_up = nx->L.sec_off[1];
            LA.nseg = nx->L.gu.nseg;
            LA.groups = nx->L.gu.groups;
            LA.codebooks = nx->L.codebooks;
            LA.stats = nx->W.stats;
            nx->pred_P = h->ahead_P;
        }
        e = launch_lut_forward(h->L, h->W, d_h, T, d_idx, d_gate, d_out, mode, recon, h->num_sms, s,
                               h->profiling ? &h->fwd_tm : nullptr, h->trace, h->trace_cap,
                               LA.keys ? &LA : nullptr);
        if (h->profiling) h->step_tm.n = 0;
    }
    if (e != cudaSuccess) return cuda_fail(e, "expert kernels");
    return ok();
}

int waste_moe_set_trace(waste_moe *h, uint64_t *d_trace, int32_t n_items) {
    if (!h) return fail(WASTE_EINVAL, "NULL handle");
    if (n_items < 0 || (n_items > 0 && !d_trace)) return fail(WASTE_EINVAL, "bad trace buffer");
    h->trace = n_items ? reinterpret_cast<unsigned long long *>(d_trace) : nullptr;
    h->trace_cap = n_items;
    return ok();
}

int waste_moe_step(waste_moe *h, const void *d_h, int32_t T, int32_t *d_idx, float *d_gate,
                   float *d_logits, float *d_out, int32_t mode, waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    int rc = check_tokens(h, T, d_h);
    if (rc) return rc;
    if (mode < 0 || mode > 2) return fail(WASTE_EINVAL, "mode = %d", mode);
    if (mode == 2 && h->cfg.act_dtype != WASTE_ACT_F32)
        return fail(WASTE_EINVAL, "mode 2 (out = h + y) needs fp32 hidden states");
    if (T == 0) return ok();
    if (!d_idx || !d_gate || !d_out) return fail(WASTE_EINVAL, "NULL idx, gate or out");
    if (!(h->cfg.flags & WASTE_FLAG_STEP_KERNEL) || use_grouped(h, T) || h->bank ||
        !fused_eligible(h->L, T, true, h->num_sms)) {
        rc = waste_moe_route(h, d_h, T, d_idx, d_gate, d_logits, stream);
        if (rc) return rc;
        return waste_moe_forward(h, d_h, T, d_idx, d_gate, d_out, mode, stream);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool recon = (h->cfg.flags & WASTE_FLAG_K2_RECONSTRUCT) != 0;
    if (h->profiling) cudaEventRecord(h->step_tm.ev[0], s);
    cudaError_t e = launch_fused_step(h->L, h->W, d_h, T, true, d_idx, d_gate,
                                      d_logits ? d_logits : h->W.logits, h->W.pred_idx, h->W.pred_count,
                                      h->pred_P > 0 ? h->pred_P : 1, d_out, mode, recon, h->num_sms, s,
                                      h->trace, h->trace_cap);
    if (h->profiling) {
        cudaEventRecord(h->step_tm.ev[1], s);
        h->step_tm.n = 2;
        h->route_tm.n = h->fwd_tm.n = 0;
    }
    if (e != cudaSuccess) return cuda_fail(e, "fused step kernel");
    return ok();
}

int waste_moe_prefetch(waste_moe *next_layer, const void *d_h, int32_t T, int32_t n_prefetch,
                       waste_stream_t side) {
    const NvtxRange nvtx_range(__func__);
    int rc = check_tokens(next_layer, T, d_h);
    if (rc) return rc;
    waste_moe *h = next_layer;
    const int P = n_prefetch < 0 ? h->lookahead : n_prefetch;
    if (P > h->L.E || P > kMaxTopK)
        return fail(WASTE_EINVAL, "n_prefetch = %d above min(n_experts, %d)", P, kMaxTopK);
    if (T == 0 || P == 0) return ok();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(side);
    cudaError_t e = launch_router(h->L, d_h, T, h->W.pred_logits, nullptr, s, h->W.router_part, h->num_sms,
                                  nullptr, nullptr, h->W.err);
    if (e != cudaSuccess) return cuda_fail(e, "lookahead router");
    e = launch_topk(h->W.pred_logits, nullptr, T, h->L.E, P, h->W.pred_idx, h->W.pred_gate_sel, nullptr,
                    nullptr, 1, nullptr, 0, s);
    if (e != cudaSuccess) return cuda_fail(e, "lookahead top-k");
    h->pred_P = P;
    if (h->bank) {
        // the predicted experts into the bank's HBM cache
        e = launch_bank_fetch(h->bank, h->bank_layer, h->W.pred_idx, T * P, false, s);
        if (e == cudaSuccess) e = launch_set_pred_count(h->W.pred_count, T, P, s);
        if (e != cudaSuccess) return cuda_fail(e, "bank lookahead");
        return ok();
    }
    e = launch_prefetch_l2(h->L, h->W.pred_idx, P, T, P, h->W.pred_count, h->W.stats, s);
    if (e != cudaSuccess) return cuda_fail(e, "L2 prefetch");
    return ok();
}

int waste_moe_set_lookahead(waste_moe *h, waste_moe *next_layer, int32_t n_prefetch) {
    const NvtxRange nvtx_range(__func__);
    if (!h) return fail(WASTE_EINVAL, "NULL handle");
    if (!next_layer || n_prefetch == 0) {
        h->ahead_next = nullptr;
        h->ahead_P = 0;
        h->ahead_routed = false;
        return ok();
    }
    if (n_prefetch < 0 || n_prefetch > next_layer->L.E || n_prefetch > kMaxTopK)
        return fail(WASTE_EINVAL, "n_prefetch = %d outside [0, min(n_experts, %d)]", n_prefetch, kMaxTopK);
    if (next_layer->L.d != h->L.d || next_layer->L.act_bf16 != h->L.act_bf16)
        return fail(WASTE_EINVAL, "the next layer's hidden size or activation type differs");
    if (next_layer->L.E > 512) return fail(WASTE_EINVAL, "the next layer has more than 512 experts");
    if (h->bank || next_layer->bank) return fail(WASTE_EINVAL, "banked layers take waste_moe_prefetch");
    h->ahead_next = next_layer;
    h->ahead_P = n_prefetch;
    h->ahead_routed = false;
    return ok();
}

int waste_moe_create_banked(const waste_moe_config *cfg, const float *d_router_w,
                            const float *d_router_bias, waste_bank *bank, int32_t layer,
                            const float *d_codebooks, waste_moe **out) {
    const NvtxRange nvtx_range(__func__);
    if (!out) return fail(WASTE_EINVAL, "out is NULL");
    *out = nullptr;
    if (!bank) return fail(WASTE_EINVAL, "NULL bank");
    int rc = check_config(cfg);
    if (rc) return rc;
    const waste_moe_config &bc = bank_config(bank);
    if (cfg->d != bc.d || cfg->f != bc.f || cfg->n_experts != bc.n_experts)
        return fail(WASTE_EINVAL, "layer shapes differ from the bank's");
    if (layer < 0 || layer >= bank_layers(bank))
        return fail(WASTE_EINVAL, "layer %d outside the bank's [0, %d)", layer, bank_layers(bank));
    // a call touches at most min(max_tokens * top_k, n_experts) distinct experts, and the plan
    // never evicts an expert of the call in flight: all of them must fit at once
    const long long per_call = std::min((long long)cfg->max_tokens * cfg->top_k, (long long)cfg->n_experts);
    if (per_call > bank_slot_count(bank))
        return fail(WASTE_EINVAL, "the bank's %d slots cannot hold the %lld distinct experts of one call",
                    bank_slot_count(bank), per_call);
    // headers (and crc with the flag) checked on the host-resident records themselves
    waste_moe *h = nullptr;
    rc = waste_moe_create(cfg, d_router_w, d_router_bias, bank_host_records(bank, layer), bank_stride(bank),
                          d_codebooks, &h);
    if (rc) return rc;
    h->bank = bank;
    h->bank_layer = layer;
    h->L.records = bank_slots(bank);
    h->L.slot_map = bank_slot_map(bank, layer);
    *out = h;
    return ok();
}

int waste_moe_stats(const waste_moe *h, waste_moe_stats_t *out) {
    if (!h || !out) return fail(WASTE_EINVAL, "NULL handle or output");
    unsigned long long v[kStatCount];
    uint32_t err = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(v, h->W.stats, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&err, h->W.err, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading statistics");
    out->demand_code_bytes = v[kStatDemandCode];
    out->codebook_bytes = v[kStatCodebook];
    out->router_bytes = v[kStatRouter];
    out->prefetch_issued_bytes = v[kStatPrefetchBytes];
    out->prefetch_experts = v[kStatPrefetchExperts];
    out->prediction_hits = v[kStatPredHits];
    out->routed_slots = v[kStatRoutedSlots];
    out->forward_slots = v[kStatForwardSlots];
    if (err & kErrTimeout) return fail(WASTE_ETIMEOUT, "a bounded device wait gave up");
    if (err & kErrNotResident)
        return fail(WASTE_EINVAL, "an expert of a banked layer had no cache slot (cache too small?)");
    if (err & kErrBadExpert) return fail(WASTE_EINVAL, "forward saw an expert index outside [0, %d)", h->L.E);
    if (err & kErrSmemLayout)
        return fail(WASTE_ECUDA, "a lookup kernel found its shared memory at another address than probed");
    return ok();
}

int waste_moe_reset_stats(waste_moe *h) {
    if (!h) return fail(WASTE_EINVAL, "NULL handle");
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemset(h->W.stats, 0, kStatCount * 8);
    if (e == cudaSuccess) e = cudaMemset(h->W.err, 0, 4);
    // a timed-out call may have left selection keys behind
    if (e == cudaSuccess) e = cudaMemset(h->W.route_slots, 0, (size_t)h->L.E * 8);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "resetting statistics");
    return ok();
}

int waste_moe_topk_from_logits(const float *d_logits, int32_t T, int32_t E, int32_t k,
                               int32_t *d_idx, float *d_gate, waste_stream_t stream) {
    if (T < 0 || E < 1 || E > kMaxExperts || k < 1 || k > E || k > kMaxTopK)
        return fail(WASTE_EINVAL, "T = %d, E = %d, k = %d out of range", T, E, k);
    if (T == 0) return ok();
    if (!d_logits || !d_idx || !d_gate) return fail(WASTE_EINVAL, "NULL pointer");
    cudaError_t e = launch_topk(d_logits, nullptr, T, E, k, d_idx, d_gate, nullptr, nullptr, 1, nullptr, 0,
                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "top-k kernel");
    return ok();
}

int waste_moe_debug_wait(waste_moe *h, const uint32_t *d_counter, uint32_t target, uint64_t limit_ns,
                         waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    if (!h) return fail(WASTE_EINVAL, "NULL handle");
    if (!d_counter || !aligned(d_counter, 4)) return fail(WASTE_EINVAL, "counter pointer NULL or not 4-byte aligned");
    if (limit_ns < 1000 || limit_ns > 10000000000ull)
        return fail(WASTE_EINVAL, "limit_ns = %llu outside [1 us, 10 s]", (unsigned long long)limit_ns);
    debug_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(d_counter, target, h->W.err,
                                                                            (unsigned long long)limit_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "wait kernel");
    return ok();
}

int waste_moe_rmsnorm(const float *d_in, float *d_out, int32_t T, int32_t d, waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    if (T < 0 || d < 1) return fail(WASTE_EINVAL, "T = %d, d = %d out of range", T, d);
    if (T == 0) return ok();
    if (!d_in || !d_out) return fail(WASTE_EINVAL, "NULL pointer");
    cudaError_t e = launch_rmsnorm(d_in, d_out, T, d, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rmsnorm kernel");
    return ok();
}

} // extern "C"
