/*
 * waste_moe.h -- C ABI of the routed-expert RVQ MoE step for NVIDIA GB300 (sm_103a).
 *
 * One handle serves one MoE layer.  Per token the layer
 *   1. computes router logits  l = W_r h (+ b),
 *   2. keeps the top-k experts (logit descending, lowest index first on equal
 *      logits) and normalises their gates with a softmax over the k selected
 *      logits,
 *   3. applies each selected expert's gate/up/down matrices straight from
 *      their residual-vector-quantised codes (3 stages, 256-entry codebooks of
 *      8-weight vectors, one uint8 code per vector and stage = 3.00 bits per
 *      weight), a = silu(G h) * (U h), y = D a, and
 *   4. adds the gate-weighted sum of the k expert outputs into the output.
 * A lookahead call runs the NEXT layer's router on the current hidden state
 * and prefetches the experts it predicts into L2; it never changes outputs.  For
 * one token it can instead ride on the current layer's step (waste_moe_set_lookahead:
 * the next layer's router rows in this layer's router launch, the prediction and
 * the prefetches in its expert launch), with no extra launch.
 *
 * Sources (web pages about the WASTE engine; page titles and sections):
 *   "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s"
 *     - "Quantification et exactitude": 3-stage RVQ, 256 entries, 8-dim
 *       vectors, 3.00 bits/weight; the matrix is never rebuilt: a table of
 *       partial dot products is built and each row costs 3 lookups + 2 adds.
 *     - "Architecture de streaming depuis le disque": one record per expert,
 *       aligned to 4 KiB, gate/up/down contiguous so one read fetches an
 *       expert; magic, expert ID and offset range are always checked;
 *       codebooks carry no checksum.
 *     - "Lecture anticipée et prédiction du routeur": 16 expert IDs per token
 *       and layer; the resident next-layer router runs on the current hidden
 *       state to prefetch 6 experts; the real router still decides, so the
 *       output is exact; total bytes read do not change; WASTE_LOOKAHEAD=0
 *       turns it off.
 *   "Chạy Kimi K3 ở 0.50 tok/s với 29GB RAM" -- the same text in Vietnamese.
 * Readings taken where the pages are silent: SwiGLU for how gate/up/down
 * combine, softmax over the selected logits, lowest-index tie-break,
 * codebooks per (expert, matrix) in fp32, the residual update h + combine.
 *
 * Conventions for every call:
 *   - Pointers named d_* are CUDA device pointers; the caller owns every
 *     buffer.  A handle BORROWS the router, records and codebooks: they must
 *     outlive it.  It owns only the workspace that create allocates and
 *     destroy frees.
 *   - Calls that take a stream only enqueue work on it and return; none
 *     synchronises the device (create and waste_moe_pack_records/stats do
 *     short synchronous copies, see each).  route/forward/prefetch allocate
 *     nothing and may be captured in a CUDA graph.
 *   - Return value: WASTE_OK (0) or a negative waste_status; the message of
 *     the last failure on the calling thread is waste_moe_last_error().
 *     Arguments are checked on the host before anything is launched; a
 *     failed check launches nothing.  Expert indices passed to forward are
 *     checked again on the device: an index outside [0, E) contributes zero
 *     and sets a sticky device error reported by waste_moe_stats as
 *     WASTE_EINVAL.
 *   - A handle is not safe for concurrent use from two host threads, and its
 *     route/forward/step calls must not run at the same time on two streams
 *     (they share the handle's workspace, including the counter by which the
 *     router's last CTA takes the top-k of a one-token call).  The lookahead
 *     goes through the next layer's handle, so it may run beside this one's.
 */
#ifndef WASTE_MOE_H
#define WASTE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WASTE_MOE_ABI_VERSION 1u

/* CUDA stream handle; ABI-identical to cudaStream_t. NULL = legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *waste_stream_t;

typedef struct waste_moe waste_moe; /* opaque; one handle per MoE layer */

typedef enum {
    WASTE_OK = 0,
    WASTE_EINVAL = -1,   /* bad argument (null pointer, size out of range, bad config) */
    WASTE_ENOMEM = -2,   /* device workspace could not be allocated */
    WASTE_ECUDA = -3,    /* a CUDA call or launch failed */
    WASTE_ELAYOUT = -4,  /* record header: bad magic / version / expert id / offset / alignment */
    WASTE_ECRC = -5,     /* record payload crc32 mismatch (WASTE_FLAG_VERIFY_CRC) */
    WASTE_ETIMEOUT = -6, /* a bounded device wait gave up */
    WASTE_ENOTIMPL = -7  /* combination the library does not implement */
} waste_status;

enum { WASTE_ACT_F32 = 0, WASTE_ACT_BF16 = 1 };

enum {
    WASTE_FLAG_VERIFY_CRC = 1u << 0,    /* create: check every record's payload crc32 */
    WASTE_FLAG_FORCE_GEMV = 1u << 2,    /* forward: table-lookup path for every slot */
    WASTE_FLAG_FORCE_MMA = 1u << 3,     /* forward: grouped dequant + tensor-core path for every
                                           call and every expert with at least one token, fp32
                                           activations included (fp16-operand accuracy) */
    WASTE_FLAG_K2_RECONSTRUCT = 1u << 4, /* forward: rebuild each 8-weight vector from the
                                            3 codebook entries in registers instead of the
                                            partial-dot-product table */
    WASTE_FLAG_STEP_KERNEL = 1u << 5, /* run forward / step as one persistent kernel that claims
                                        router, top-k, expert and combine work from a device
                                        queue, instead of one kernel per phase (same results,
                                        bit for bit) */
    WASTE_FLAG_BANK_SERIAL = 1u << 6  /* banked layers: copy a call's missing experts first and
                                        run the expert kernels after, instead of consuming each
                                        expert as its copy lands (same results, bit for bit) */
};

/* Layer configuration.  d % 8 == 0, f % 8 == 0, 1 <= top_k <= n_experts <= 4096,
 * top_k <= 32, 1 <= max_tokens.  lookahead = experts predicted per token by
 * waste_moe_prefetch when its n_prefetch is negative (the pages use 6; 0 = off);
 * the environment variable WASTE_LOOKAHEAD, when set, overrides it at create. */
typedef struct {
    uint32_t abi_version; /* must equal WASTE_MOE_ABI_VERSION */
    int32_t d;            /* hidden size */
    int32_t f;            /* expert FFN width */
    int32_t n_experts;    /* E */
    int32_t top_k;        /* k */
    int32_t act_dtype;    /* WASTE_ACT_F32 or WASTE_ACT_BF16: dtype of the hidden states h */
    int32_t max_tokens;   /* largest T passed to route/forward/prefetch (sizes the workspace) */
    int32_t lookahead;    /* default prefetch count */
    uint32_t flags;       /* WASTE_FLAG_* */
    int32_t layer;        /* layer id expected in the record headers; -1 = do not check */
} waste_moe_config;

/* ---- record format -------------------------------------------------------------------
 * The experts of a layer form a bank of records of equal stride (a multiple of
 * 4096 B), record e at byte e * stride of the bank, the bank 4096-aligned.  A record
 * is a 4096 B header followed by three sections (gate, up, down), each starting on a
 * 4096 B boundary, holding that matrix's codes in the tiled order below.
 *
 * Code tiling of one matrix with n_out rows and n_in = 8 nv inputs (vector j of row r
 * covers inputs 8j .. 8j+7; codes code[r][s][j], s = stage):
 *   segments  sigma = 0 .. ceil(nv/32)-1  (32 vectors each),
 *   row groups g    = 0 .. ceil(n_out/16)-1 (16 rows each),
 *   16-byte chunk (sigma, g, s, jj) at byte ((sigma*G + g)*3 + s)*512 + jj*16,
 *   byte q of that chunk = code[16g + ((jj ^ q) & 15)][s][32 sigma + jj]
 *   (0 where the row or vector is past the end).
 * The xor spreads each lane's 16 rows so the table-lookup kernel can reduce
 * across lanes without selects; the order is a fixed part of the format. */
#define WASTE_RECORD_MAGIC 0x454F4D57u /* bytes "WMOE" */
#define WASTE_RECORD_VERSION 1u
#define WASTE_RECORD_ALIGN 4096u
#define WASTE_LAYOUT_TILED16X 1u

typedef struct {
    uint32_t magic;              /* WASTE_RECORD_MAGIC */
    uint32_t version;            /* WASTE_RECORD_VERSION */
    int32_t layer;               /* layer id written by pack */
    int32_t expert_id;           /* must equal the record's index in the bank */
    int32_t d, f;                /* shapes the codes were written for */
    int32_t n_stages;            /* 3 */
    int32_t codebook_size;       /* 256 */
    int32_t vec;                 /* 8 */
    uint32_t layout_id;          /* WASTE_LAYOUT_TILED16X */
    uint64_t section_offset[3];  /* gate, up, down: byte offset from the record start */
    uint64_t section_bytes[3];   /* bytes of each section (multiple of 4096) */
    uint64_t record_bytes;       /* stride the record was written for */
    uint32_t payload_crc32;      /* crc32 (IEEE, reflected 0xEDB88320) of the three
                                    sections in order; 0 = not computed */
    uint32_t reserved;
} waste_record_header;

/* Layout of one record for cfg: the minimal stride and the three sections.
 * Pure host arithmetic; any output pointer may be NULL. */
int waste_moe_record_layout(const waste_moe_config *cfg, size_t *record_stride,
                            size_t section_offset[3], size_t section_bytes[3]);

/* Write records [expert_begin, expert_begin + n_experts) of a bank from codes in
 * the logical layout (the converter's last step):
 *   d_gate_codes, d_up_codes: [n_experts][f][3][d/8] uint8,
 *   d_down_codes:             [n_experts][d][3][f/8] uint8  (device, read only).
 * d_records is the bank base (4096-aligned); record_stride as above.  Headers
 * carry `layer`.  Enqueued on stream.  With compute_crc != 0 the payload crc32 of each
 * record (IEEE 802.3 / zlib crc32 of the three sections in order) is computed on the
 * device and stored in its header; the call then allocates a temporary device buffer
 * (4 bytes per 4 KiB of payload) and waits for the stream. */
int waste_moe_pack_records(const waste_moe_config *cfg, int32_t layer, int32_t expert_begin,
                           int32_t n_experts, const uint8_t *d_gate_codes,
                           const uint8_t *d_up_codes, const uint8_t *d_down_codes,
                           uint8_t *d_records, size_t record_stride, int32_t compute_crc,
                           waste_stream_t stream);

/* Create a handle for one layer.
 *   d_router_w    [E][d] fp32 router weights (borrowed)
 *   d_router_bias [E] fp32 or NULL (borrowed)
 *   d_records     bank of E records, 4096-aligned base, stride record_stride (borrowed)
 *   d_codebooks   [E][3 matrices: gate, up, down][3 stages][256][8] fp32 (borrowed)
 * Checks every record header (magic, version, expert id, layer, shapes, section
 * offsets inside the stride and 4096-aligned, sizes) with one synchronous copy of
 * the headers.  With WASTE_FLAG_VERIFY_CRC it also recomputes every record's payload
 * crc32 on the device (page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section
 * "Architecture de streaming depuis le disque": crc32 behind --verify) and refuses a
 * record whose header holds 0 or a different value (WASTE_ECRC).  On any failure
 * returns < 0 and sets *out = NULL (the layer is refused rather than run on
 * suspect weights).  Allocates the workspace (sized by max_tokens). */
int waste_moe_create(const waste_moe_config *cfg, const float *d_router_w,
                     const float *d_router_bias, const uint8_t *d_records,
                     size_t record_stride, const float *d_codebooks, waste_moe **out);

/* Route T tokens (0 <= T <= max_tokens; T == 0 does nothing).
 *   d_h      [T][d] hidden states, fp32 or bf16 per act_dtype
 *   d_idx    [T][k] int32 out: selected experts in rank order
 *   d_gate   [T][k] fp32 out: softmax of the selected logits
 *   d_logits [T][E] fp32 out, or NULL (then kept in the workspace)
 * If waste_moe_prefetch ran for this layer (ordered before this call by the
 * caller), the number of predicted experts among the selected ones is added to
 * the prediction_hits statistic.  One token (T == 1) is routed in one launch whose
 * CTAs move their rows of W_r and the token into shared memory with bulk copies;
 * a copy that does not land within a bounded wait (about a second) leaves the
 * outputs undefined and makes waste_moe_stats return WASTE_ETIMEOUT. */
int waste_moe_route(waste_moe *h, const void *d_h, int32_t T, int32_t *d_idx, float *d_gate,
                    float *d_logits, waste_stream_t stream);

/* Apply the selected experts and combine (0 <= T <= max_tokens).
 *   d_h      [T][d] hidden states (fp32 or bf16 per act_dtype)
 *   d_idx    [T][k] int32, d_gate [T][k] fp32 (usually route's outputs)
 *   d_out    [T][d] fp32, any memory the device can write: device memory, or pinned
 *            (or, where the GPU addresses it, any) host memory, which the combine then
 *            writes over the CPU-GPU link with no separate copy
 *   mode 0: out  = sum_i gate_i * y_i
 *   mode 1: out += sum_i gate_i * y_i   (residual already in out)
 *   mode 2: out  = h + sum_i gate_i * y_i (fp32 h only; out may equal h)
 * Deterministic: the same inputs give bit-identical outputs (fixed summation
 * order, no floating-point atomics).
 * Batched calls (bf16 activations and T > 1, or WASTE_FLAG_FORCE_MMA): the slots are
 * grouped by expert on the device; every expert chosen by at least 4 tokens of the
 * call (environment WASTE_MMA_MIN_TOKENS overrides 4; 1 under WASTE_FLAG_FORCE_MMA)
 * is applied as a dense product on the tensor cores -- 128-row tiles of its codes
 * decoded into fp16 weights in shared memory, its tokens' activations as fp16,
 * fp32 accumulation -- and the other slots take the table-lookup path.  The page
 * "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée et
 * prédiction du routeur", puts one layer of a prefill chunk at about 550 expert
 * slots: many tokens per expert.  Tensor-core slots carry fp16-operand error
 * (relative L2 about 1e-3 at most on the output); WASTE_FLAG_FORCE_GEMV keeps every
 * slot on the fp32 lookup path. */
int waste_moe_forward(waste_moe *h, const void *d_h, int32_t T, const int32_t *d_idx,
                      const float *d_gate, float *d_out, int32_t mode, waste_stream_t stream);

/* route + forward in one call: d_idx, d_gate (and d_logits if not NULL) receive the
 * routing, d_out the combined output per mode (as waste_moe_forward).  With
 * WASTE_FLAG_STEP_KERNEL (and shapes that allow it: E <= 1024) it runs as one persistent
 * kernel; otherwise as route then forward.  Results are identical either way. */
int waste_moe_step(waste_moe *h, const void *d_h, int32_t T, int32_t *d_idx, float *d_gate,
                   float *d_logits, float *d_out, int32_t mode, waste_stream_t stream);

/* Trace work items into d_trace (4 uint64 per item, %globaltimer in ns).
 * Persistent step kernel: item i in queue order (router items, the top-k item, gate/up
 * units, down units, combine items) writes {start, end, SM id, CTA index}.
 * Per-phase kernels: lookup unit i (gate/up units, then down units) writes
 * {start, tables built, end, SM id | (ns from start to the barrier before the table
 * build) << 32}.
 * n_items = capacity in items; 0 (or d_trace NULL with 0) turns it off.  The buffer is the
 * caller's and must outlive the traced calls. */
int waste_moe_set_trace(waste_moe *h, uint64_t *d_trace, int32_t n_items);

/* Lookahead: run next_layer's router on the current hidden states d_h [T][d],
 * take its top n_prefetch experts per token (n_prefetch < 0: the handle's
 * lookahead; 0: nothing) and prefetch into L2 what their gate/up units read
 * first: the first 16 row groups of every 32-vector segment of gate and up, and
 * the gate and up codebooks (about 1.4 MB per expert at d = 7168, f = 1536; the
 * whole record would not survive the current layer's stream in L2).  On a
 * banked handle the predicted records are copied into the HBM cache instead.
 * Writes no user-visible buffer and never changes any output.  The caller orders it after
 * d_h is ready and before next_layer's route (events), and must not overwrite
 * d_h until it has run. */
int waste_moe_prefetch(waste_moe *next_layer, const void *d_h, int32_t T, int32_t n_prefetch,
                       waste_stream_t side);

/* Lookahead inside the step (page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section
 * "Lecture anticipée et prédiction du routeur": layer L+1's router runs on layer L's input and its
 * top experts are fetched ahead), for one-token calls on resident layers, with no extra launch
 * and no side stream.  After this call, a one-token waste_moe_route on h also runs next_layer's
 * router rows on the same input (the extra rows ride on h's router launch), and the
 * waste_moe_forward that follows it (or waste_moe_step) takes next_layer's top n_prefetch experts
 * from those logits -- the order of next_layer's own top-k -- as its prediction (scored by
 * next_layer's next route, as after waste_moe_prefetch) and asks L2 for the same pieces as
 * waste_moe_prefetch, from the CTAs of h's expert kernel that have no down unit once their
 * gate/up units are done.  Outputs and demand bytes are unchanged.  next_layer = NULL or
 * n_prefetch = 0 turns it off.  Errors: WASTE_EINVAL for NULL h, n_prefetch outside
 * [0, min(n_experts, 32)], a next layer with another hidden size or activation type or more than
 * 512 experts, or banked handles (they take waste_moe_prefetch).  A call whose shapes do not
 * allow it (several tokens, a router launch that would not fit with the extra rows) runs without
 * it.  h's step and next_layer's route must be ordered on one stream (or by events); h keeps a
 * pointer to next_layer, which must stay alive while the setting holds (turn it off, or destroy
 * h, first). */
int waste_moe_set_lookahead(waste_moe *h, waste_moe *next_layer, int32_t n_prefetch);

/* Free the workspace and the handle (NULL is ignored).  Synchronises the device. */
void waste_moe_destroy(waste_moe *h);

typedef struct {
    uint64_t demand_code_bytes;     /* code bytes the expert kernels read (algorithmic) */
    uint64_t codebook_bytes;        /* codebook bytes used by the expert kernels */
    uint64_t router_bytes;          /* router weight bytes read by route */
    uint64_t prefetch_issued_bytes; /* record and codebook bytes named in L2 prefetches */
    uint64_t prefetch_experts;      /* (token, expert) prefetches issued */
    uint64_t prediction_hits;       /* routed experts that had been predicted */
    uint64_t routed_slots;          /* (token, expert) slots routed */
    uint64_t forward_slots;         /* (token, expert) slots applied by forward */
} waste_moe_stats_t;

/* Copy the handle's counters (one synchronous copy on the legacy stream after a
 * device synchronise).  Returns WASTE_ETIMEOUT if a bounded device wait gave up,
 * WASTE_EINVAL if a kernel saw an expert index out of range (since create or the
 * last reset), else WASTE_OK.  After WASTE_ETIMEOUT the outputs of the calls since the
 * last reset are not to be used, and the context is to be treated as unusable: a kernel
 * that gave up may have left asynchronous copies or tensor-core operations behind it. */
int waste_moe_stats(const waste_moe *h, waste_moe_stats_t *out);

/* Zero the counters (synchronous). */
int waste_moe_reset_stats(waste_moe *h);

/* Per-kernel timing of the following route/forward calls with CUDA events recorded
 * on the call's stream (enable != 0 creates the events, 0 drops them; do not enable
 * while a stream is being captured into a graph). */
int waste_moe_set_profiling(waste_moe *h, int32_t enable);

/* Milliseconds of each kernel of the last profiled calls: ms[0] router, ms[1] top-k
 * (route; -1 where the router's last CTA took the top-k); ms[2] gate/up, ms[3] down, ms[4] combine (forward as separate kernels; where
 * the gate/up and down units ran in one launch, ms[2] is that launch and ms[3] is -1);
 * ms[5] the persistent step kernel (step, or forward when fused); -1 where the last
 * call did not run that kernel.  Waits for the events. */
int waste_moe_read_profile(const waste_moe *h, float ms[6]);

/* ---- Tiered expert bank ---------------------------------------------------------
 * Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", sections "Budget RAM et zone de
 * performance étroite" and "Lecture anticipée et prédiction du routeur": the experts live
 * in a large slow tier, a bounded cache holds some of them, a miss reads the expert's
 * record from the slow tier, and the next layer's router fills the cache ahead of demand.
 * Here the slow tier is host memory (pinned, read by the GPU) and the cache is HBM.  The
 * fetch runs on the device: a plan (every requested expert already in the cache takes the
 * call's stamp; each miss then takes the least recently used slot not stamped by the call in
 * flight) and a copy of the missing records. */
typedef struct waste_bank waste_bank;

typedef struct {
    uint64_t demand_hits;      /* (token, expert) slots whose expert was in the cache when its
                                  layer ran (or brought in earlier in the same call) */
    uint64_t demand_misses;    /* experts copied in on demand */
    uint64_t prefetch_copies;  /* experts copied in by a lookahead */
    uint64_t prefetch_present; /* predicted experts already in the cache */
    uint64_t copied_bytes;     /* host -> HBM bytes (demand and lookahead) */
} waste_bank_stats_t;

/* n_layers x cfg->n_experts records (written by waste_moe_pack_records into device memory,
 * then copied out) in host memory the device can read -- pinned (cudaHostAlloc,
 * cudaMallocHost, cudaHostRegister), or any host memory on systems whose GPU addresses it
 * directly; cudaHostGetDevicePointer decides (WASTE_EINVAL when it refuses): layer L's
 * expert e at host_records + (L * n_experts + e) * record_stride, host_records 4096-aligned
 * (WASTE_ELAYOUT).  n_slots records of HBM cache.  The records are borrowed; the cache is
 * the bank's own. */
int waste_bank_create(const waste_moe_config *cfg, int32_t n_layers, const uint8_t *host_records,
                      size_t record_stride, int32_t n_slots, waste_bank **out);
void waste_bank_destroy(waste_bank *bank);
/* Empty the cache and zero the counters (synchronous). */
int waste_bank_reset(waste_bank *bank);
int waste_bank_stats(const waste_bank *bank, waste_bank_stats_t *out);

/* A layer handle whose expert records are layer `layer` of a bank (headers -- and the payload
 * crc32 with WASTE_FLAG_VERIFY_CRC -- checked as by waste_moe_create).  forward / step first
 * fetch the routed experts into the cache, then read them from their slots; prefetch copies
 * the predicted experts into the cache instead of warming L2.  Outputs equal those of the
 * same records held in device memory, bit for bit.  Needs n_slots >= min(max_tokens * top_k,
 * n_experts), the most distinct experts one call can touch (WASTE_EINVAL otherwise).
 * A call on the table-lookup path with T * top_k <= 64 (decode) runs its demand copy inside
 * the persistent step kernel: a few CTAs copy the missing records in order while the others
 * run the resident experts' units and then each missing expert's as soon as its record is in
 * (page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée et
 * prédiction du routeur": the compute consumes each expert as it arrives);
 * WASTE_FLAG_BANK_SERIAL turns this off.
 * The fetches of one bank are ordered by events the bank holds, on whatever streams they are
 * issued: each demand fetch waits for the bank's last lookahead fetch, and each lookahead
 * fetch for the last demand fetch (its plan, when the copy runs in the step kernel; a
 * lookahead never evicts an expert of the call in flight).  Issue a layer's forward before
 * the lookahead into the next layer, so that the lookahead's copies run beside the forward.
 * These waits use events recorded by earlier calls, so banked layers are not for stream
 * capture into CUDA graphs. */
int waste_moe_create_banked(const waste_moe_config *cfg, const float *d_router_w,
                            const float *d_router_bias, waste_bank *bank, int32_t layer,
                            const float *d_codebooks, waste_moe **out);

/* ---- RVQ encoder (the step before the path) -------------------------------------------
 * Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Quantification et
 * exactitude": expert matrices are stored as 3 residual stages of 256 eight-dimensional
 * vectors; the converter that writes them is named there, its training is not.  This one is
 * greedy residual k-means: the residual R starts as W; per stage s, centroid c starts as the
 * residual vector d_init[s][c]; `iters` Lloyd rounds assign every vector to its nearest
 * centroid and move each centroid with members to their mean (an empty one stays); a last
 * assignment gives the stage's codes and R -= C[code].  Nearest = least sum over v = 0..7 of
 * (x_v - c_v)^2 in fp32, in that order, one fused multiply-add per term, ties to the lower
 * index; means are taken from exact fixed-point sums (round(x * 2^40) as int64):
 * mean = (float)((sum / count) * 2^-40) in double.  Codes and codebooks are therefore the same
 * on every run and equal to any implementation of these rules.
 *
 * d_w [rows][cols] fp32 row-major (device), cols % 8 == 0, every |w| < 2^22 and finite
 * (WASTE_EINVAL otherwise); vector j of row r covers columns 8j..8j+7 and is vector r*(cols/8)+j.
 * d_init [3][256] int32 vector indices in [0, rows*cols/8) (WASTE_EINVAL otherwise); iters >= 0.
 * Outputs (device, caller-owned): d_codebooks [3][256][8] fp32, d_codes [rows][3][cols/8] uint8
 * (the logical layout waste_moe_pack_records reads), d_err [3] double = sum of the squared
 * residual components after each stage.  Synchronous on `stream`; allocates and frees its own
 * scratch (rows*cols*4 bytes plus 18 KiB). */
int waste_rvq_train(const float *d_w, int32_t rows, int32_t cols, const int32_t *d_init, int32_t iters,
                    float *d_codebooks, uint8_t *d_codes, double *d_err, waste_stream_t stream);
/* The three final assignments alone, with given codebooks d_codebooks [3][256][8]. */
int waste_rvq_encode(const float *d_w, int32_t rows, int32_t cols, const float *d_codebooks, uint8_t *d_codes,
                     double *d_err, waste_stream_t stream);

/* Message of the last failure on the calling thread ("" if none). */
const char *waste_moe_last_error(void);

/* Top-k + softmax of given logits (the routing step alone; used by tests to
 * drive exact ties).  d_logits [T][E] fp32, d_idx/d_gate [T][k]. */
int waste_moe_topk_from_logits(const float *d_logits, int32_t T, int32_t E, int32_t k,
                               int32_t *d_idx, float *d_gate, waste_stream_t stream);

/* Weightless RMS normalisation of T rows of d floats: out = in / sqrt(mean(in^2) + 1e-6)
 * (out may equal in).  Not one of the pages' operations: it stands in for the
 * normalisation a model's trunk applies to each MoE layer's input, so that a stack of
 * layers driven by h += combine keeps its inputs at unit scale. */
int waste_moe_rmsnorm(const float *d_in, float *d_out, int32_t T, int32_t d, waste_stream_t stream);

/* Test aid for the refusal path of the library's device waits.  Work items of the
 * persistent step kernel wait on one another through device counters (thread 0 polls with
 * acquire loads and a growing sleep, then its CTA proceeds); every such wait is bounded, and
 * one that gives up latches a timeout in the handle's error word, which waste_moe_stats
 * reports as WASTE_ETIMEOUT (the pages' rule: refuse rather than degrade, page "Exécuter
 * Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Budget RAM et zone de performance
 * étroite").  This call runs that same wait, in one CTA on `stream`, on a counter the caller
 * owns: it returns once *d_counter >= target, or after limit_ns nanoseconds (1 us .. 10 s)
 * with the timeout latched in h.  A test withholds the counter to see the refusal without
 * hanging or faulting the GPU; the context stays usable.  The library never calls it.
 *   d_counter   device (or device-accessible) uint32, 4-byte aligned; only read
 * Returns WASTE_EINVAL for a NULL handle or counter or a limit outside the range. */
int waste_moe_debug_wait(waste_moe *h, const uint32_t *d_counter, uint32_t target, uint64_t limit_ns,
                         waste_stream_t stream);

/* waste_moe_forward without a handle and without allocating anything.
 *
 * The pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory -- for example a host that only receives device pointers
 * from an engine which owns all of the GPU's memory, or code running where
 * cudaMalloc is not allowed.  It always runs the fp32 table-lookup kernels on the
 * same records, codebooks, hidden states, experts and gates, and keeps its partial
 * sums in one fixed 8 MiB array inside the library's device image (every GPU that
 * loads the library holds it until the process exits).  Its output therefore equals
 * waste_moe_forward's within the fp32 bar wherever the handle's forward also runs the
 * lookup kernels (fp32 hidden states, one token, or WASTE_FLAG_FORCE_GEMV); for a
 * batched bf16 call, whose experts with several tokens the handle's forward sends to
 * the fp16 tensor-core path, the two agree only to the bf16 bar (relative L2 2e-3).
 *   cfg          shapes and act_dtype (d, f, n_experts, top_k, act_dtype, flags as
 *                for create; max_tokens, lookahead and layer are ignored)
 *   d_records    bank of records, 4096-aligned; not re-validated here (validate
 *                once, e.g. with waste_moe_create)
 *   d_codebooks, d_h, d_idx, d_gate, d_out, mode: as for waste_moe_forward
 * Limits: the T * top_k slots need (f * 2 * ceil(d/512) + d * ceil(f/512)) * 4 bytes
 * of scratch each (about 0.26 MB at d = 7168, f = 1536, i.e. T * top_k <= 32 there);
 * a call beyond 8 MiB in total is rejected with WASTE_EINVAL and launches nothing.
 * No cudaMalloc, cudaFree or other allocating routine is called.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) once for that device; make that first call before any
 * stream capture.  Every call shares the one array, so calls that overlap on the
 * GPU (other streams, other threads) race and give wrong results: serialise them.
 * An expert index outside [0, E) contributes zero; it is not reported here. */
int waste_moe_forward_noalloc(const waste_moe_config *cfg, const uint8_t *d_records,
                              size_t record_stride, const float *d_codebooks, const void *d_h,
                              int32_t T, const int32_t *d_idx, const float *d_gate, float *d_out,
                              int32_t mode, waste_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* WASTE_MOE_H */
