// Internal declarations shared by the translation units of libwaste_moe.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>

#include "waste_moe.h"

namespace wm {

constexpr int kStages = 3;
constexpr int kCodes = 256;
constexpr int kVec = 8;
constexpr int kSegVec = 32;    // vectors per segment (one per lane)
constexpr int kGroupRows = 16; // rows per 16-byte chunk
constexpr int kMaxExperts = 4096;
constexpr int kMaxTopK = 32;
constexpr int kMaxFusedRowBlocks = 64; // down row blocks the fused step kernel can track

// Sticky device error bits.
enum : uint32_t { kErrBadExpert = 1u, kErrTimeout = 2u, kErrNotResident = 4u, kErrSmemLayout = 8u };

// Record of expert e: by index, or through a bank's slot map (null when the expert has no
// slot -- the caller treats it as an invalid expert).
__device__ __forceinline__ const uint8_t *expert_record(const uint8_t *records, size_t stride,
                                                        const int32_t *slot_map, int e) {
    if (!slot_map) return records + (size_t)e * stride;
    const int s = slot_map[e];
    return s >= 0 ? records + (size_t)s * stride : nullptr;
}

// Device counters, indices into the handle's uint64 counter array.
enum {
    kStatDemandCode = 0,
    kStatCodebook,
    kStatRouter,
    kStatPrefetchBytes,
    kStatPrefetchExperts,
    kStatPredHits,
    kStatRoutedSlots,
    kStatForwardSlots,
    kStatCount
};

// Geometry of one tiled matrix section.
struct MatGeom {
    int n_out, n_in;
    int nv;     // vectors per row
    int nseg;   // 32-vector segments
    int groups; // 16-row groups
    __host__ __device__ size_t chunk_bytes() const { return (size_t)nseg * groups * kStages * 512; }
};

inline MatGeom mat_geom(int n_out, int n_in) {
    MatGeom g;
    g.n_out = n_out;
    g.n_in = n_in;
    g.nv = n_in / kVec;
    g.nseg = (g.nv + kSegVec - 1) / kSegVec;
    g.groups = (n_out + kGroupRows - 1) / kGroupRows;
    return g;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Devices the per-device host caches below track (ordinals past it are served uncached).
constexpr int kMaxDevices = 64;

// The dynamic shared memory a kernel may ask for is an attribute of the kernel on each
// device: it is set on the current device the first time a launcher needs `bytes` there
// (a cheap driver call; the cache only avoids repeating it).  One SmemAttr per kernel.
struct SmemAttr {
    std::atomic<int> bytes[kMaxDevices] = {};
};
inline cudaError_t ensure_smem(SmemAttr &a, const void *kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached && a.bytes[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && cached) a.bytes[dev].store(bytes, std::memory_order_release);
    return e;
}

// Everything a kernel needs to reach one layer's weights.
struct LayerView {
    const float *router_w;
    const float *router_b;
    const uint8_t *records;   // record of expert e at records + e * stride, or (slot_map)
    const int32_t *slot_map;  // optional [E]: record of expert e at records + slot_map[e] * stride
    size_t stride;
    size_t sec_off[3];
    const float *codebooks; // [E][3][3][256][8]
    int d, f, E, k;
    int act_bf16;
    MatGeom gu;   // gate / up geometry (f rows, d inputs)
    MatGeom dn;   // down geometry (d rows, f inputs)
};

// Device state of a tiered expert bank (see bank.cu).
struct BankDevice {
    void *base;
    uint8_t *slots;       // [n_slots] records in HBM
    int32_t *map;         // [n_layers * E] (layer, expert) -> slot, or -1
    int32_t *key_of;      // [n_slots] slot -> layer * E + expert, or -1
    uint32_t *tick;       // [n_slots] clock of the last call that used the slot
    int2 *jobs;           // [n_slots] copy jobs of the last plan: (slot, key)
    uint32_t *job_seq;    // [n_slots] plan that last made the slot a copy job
    int32_t *job_of;      // [n_slots] its job index in that plan
    uint32_t *clock;      // advanced by every demand fetch
    int32_t *n_jobs;
    uint32_t *seq;        // advanced by every plan
    unsigned long long *stats;
};
// The copy of a demand fetch run by the persistent step kernel beside the expert units:
// lanes CTAs copy the plan's jobs chunk by chunk, and every unit of a slot whose record is
// being copied (wait_job[slot] >= 0) waits for that job's chunks first.
struct BankLanes {
    BankDevice D;
    const uint8_t *host; // device-usable address of the host records
    const int32_t *wait_job; // [slots] job the slot's record arrives by, or -1
    int lanes;
};
enum { kBankDemandHits = 0, kBankDemandMisses, kBankPrefetchCopies, kBankPrefetchPresent, kBankCopiedBytes,
       kBankStatCount };

// Top-k taken by the last CTA of the router launch (router.cu); done = null: router only.
struct RouteTopk {
    unsigned *done; // CTAs finished, zero at rest
    int k;
    int32_t *idx;
    float *gate;
    const int32_t *pred_idx;
    int32_t *pred_count;
    int pred_stride;
    unsigned long long *stats;
    unsigned long long router_bytes;
    unsigned long long *slots; // [E] one-token router: each expert's selection key, 0 at rest
    // optional, polled one-token router only: the next layer's router rows on the same input
    // (ahead_E experts, weights ahead_w, bias ahead_b), whose selection keys go to ahead_keys
    const float *ahead_w, *ahead_b;
    int ahead_E;
    unsigned long long *ahead_keys;
};

// L2 prefetch of a predicted expert (the lookahead).  With every expert resident in HBM the only
// gain is the first read of each unit, so the lookahead asks L2 for what the gate/up units of
// the expert read first -- the first kLookaheadGroups row groups of each 32-vector segment of
// gate and up (one round of a 16-warp unit's row stream) -- and the expert's gate and up
// codebooks: about 1.4 MB per expert at d = 7168, f = 1536, small enough to stay in L2 while the
// current layer streams, where whole records (12.4 MB each) were evicted before use and read
// twice.  Piece i of an expert: the segments of gate (i < nseg) and up, then the codebooks.
constexpr int kLookaheadGroups = 16;
constexpr uint32_t kLookaheadCbBytes = 2 * kStages * kCodes * kVec * 4; // gate and up codebooks

__host__ __device__ inline int lookahead_pieces(int nseg) { return 2 * nseg + 1; }
__host__ __device__ inline unsigned long long lookahead_bytes(int nseg, int groups) {
    const int g = groups < kLookaheadGroups ? groups : kLookaheadGroups;
    return (unsigned long long)2 * nseg * (unsigned long long)(g * (kStages * 512)) + kLookaheadCbBytes;
}
#ifdef __CUDACC__
__device__ __forceinline__ void lookahead_piece(const uint8_t *records, size_t stride, size_t off_gate,
                                                size_t off_up, int nseg, int groups, const float *codebooks,
                                                int e, int i) {
    if (i < 2 * nseg) {
        const uint32_t seg_bytes = (uint32_t)min(groups, kLookaheadGroups) * (kStages * 512);
        const uint8_t *q = records + (size_t)e * stride + (i < nseg ? off_gate : off_up) +
                           (size_t)(i % nseg) * groups * (kStages * 512);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(q), "r"(seg_bytes) : "memory");
    } else {
        const float *cb = codebooks + (size_t)e * 3 * kStages * kCodes * kVec;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(cb), "r"(kLookaheadCbBytes) : "memory");
    }
}
#endif

// Slots of a batched call grouped by expert (see grouped.cu).
struct Grouping {
    int32_t *offs;      // [E + 1] first position of each expert in `sorted`
    int32_t *sorted;    // [max_slots] slots grouped by expert, ascending within an expert
    int32_t *lut_slots; // [max_slots] slots left to the lookup kernels, ascending
    int4 *chunks;       // [max_chunks] (expert, first position in sorted, tokens, first tile row)
    int32_t *counts;    // [2] chunks, lookup slots
    uint8_t *one_part;  // [max_slots] 1: the slot's down output is partial 0 alone
    uint8_t *xg;        // fp16 activation tiles of the chunks (gate/up input), rows x ceil(d/64) x 128 B
    uint8_t *ag;        // fp16 SwiGLU tiles of the chunks (down input), rows x ceil(f/64) x 128 B
    int max_chunks;
};
// Tile rows the grouped path needs at most (tokens padded to 16 per chunk).
size_t grouped_tile_rows(int max_slots, int max_chunks);

struct Workspace {
    float *logits;       // [max_T][E]
    float *logits_lo;    // [max_T][E]
    float *pred_logits;  // [max_T][E]
    int32_t *pred_idx;   // [max_T][kMaxTopK]
    int32_t *pred_count; // [max_T]
    int32_t *pred_idx_sel; // scratch for prefetch top-k
    float *pred_gate_sel;  // scratch (unused gates of the prediction)
    float *part_gu;      // [max_slots][(gu.nseg + 1) / 2][2][f]
    float *part_dn;      // [max_slots][(dn.nseg + 1) / 2][d]; tensor-core slots use part 0
    unsigned long long *stats; // [kStatCount]
    uint32_t *err;       // sticky error bits
    unsigned *sync;      // fused-step queue and counters [4 + 2 max_slots + kMaxFusedRowBlocks], zero at rest
    int32_t *bank_wait;  // [max_slots] banked calls: job each slot's record arrives by, or -1
    int32_t *bank_order; // [max_slots] banked calls: slots in the order their units run
    unsigned *route_done; // router CTAs finished (the router launch that also takes the top-k)
    unsigned long long *route_slots; // [E] one-token router's selection keys, zero at rest
    unsigned long long *ahead_keys;  // [E] this layer's selection keys from the previous layer's router launch
    Grouping grp;        // batched calls only (null pointers when max_tokens == 1)
    float *router_part;  // [kRouterMaxSplits][max_T][E] when max_T > 16, else null
    void *base;
    size_t bytes;
};

// ---- launchers (each returns cudaGetLastError() of its launches) ----
// logits_lo (optional): exact remainder of adding the router bias, so that
// logits + logits_lo equals W_r h + b exactly given the fp32 dot product.
// part (optional): [kRouterMaxSplits][T][E] scratch for the split-K router of T > 16.
constexpr int kRouterMaxSplits = 32;
// With fuse (and T == 1): the router's last CTA also takes the top-k, and *fused says so
// (else the caller launches the top-k).  err (optional): sticky device error bits (a bounded
// wait that gave up sets kErrTimeout).
cudaError_t launch_router(const LayerView &L, const void *h, int T, float *logits,
                          float *logits_lo, cudaStream_t s, float *part = nullptr, int num_sms = 1,
                          const RouteTopk *fuse = nullptr, bool *fused = nullptr, uint32_t *err = nullptr);
// Whether the polled one-token router fits with ahead_E more expert rows (the next layer's).
bool route_polled_fits(const LayerView &L, const void *h, int T, int ahead_E, int num_sms);
cudaError_t launch_topk(const float *logits, const float *logits_lo, int T, int E, int k,
                        int32_t *idx, float *gate, const int32_t *pred_idx, int32_t *pred_count,
                        int pred_stride, unsigned long long *stats,
                        unsigned long long router_bytes, cudaStream_t s);
// Optional per-kernel timing: events[i] is recorded after the i-th kernel (events[0] before
// the first); null = no timing.
struct Timing {
    cudaEvent_t ev[8];
    int n;
};
// The lookahead inside a one-token expert launch: the next layer's top-P experts, chosen from the
// selection keys its router rows produced in this layer's router launch (same input), and their
// first pieces asked of L2 (lookahead_piece) by the CTAs that have no down unit, once their
// gate/up units are done.
struct LutAhead {
    const unsigned long long *keys; // [E] the next layer's selection keys; null: no lookahead
    int E, P;
    int32_t *pred_idx, *pred_count;  // the next layer's prediction (P experts, rank order)
    const uint8_t *records;          // the next layer's records and codebooks
    size_t stride, off_gate, off_up;
    int nseg, groups;
    const float *codebooks;
    unsigned long long *stats;       // the next layer's counters (prefetched bytes and experts)
};
// trace (optional): per-unit trace of the two lookup kernels, trace_cap units.  ahead
// (optional): the lookahead of a one-token call (taken by the one-launch expert kernel only).
cudaError_t launch_lut_forward(const LayerView &L, const Workspace &W, const void *h, int T,
                               const int32_t *idx, const float *gate, float *out, int mode,
                               bool reconstruct, int num_sms, cudaStream_t s, Timing *tm,
                               unsigned long long *trace = nullptr, int trace_cap = 0,
                               const LutAhead *ahead = nullptr);
// Down partials per slot written by the lookup kernels (one per pair of segments).
inline int down_parts(const LayerView &L) { return (L.dn.nseg + 1) / 2; }
// One lookup phase (gate/up or down) over the slots listed on the device.
cudaError_t launch_lut_listed(const LayerView &L, const Workspace &W, const void *h, int T,
                              const int32_t *idx, const int32_t *slot_list, const int32_t *n_list,
                              bool down, bool reconstruct, int num_sms, cudaStream_t s);
// out = / += / h + sum_i gate * (sum of the slot's down partials); one_part (optional)
// marks slots whose output is partial 0 alone.
cudaError_t launch_combine(const LayerView &L, const Workspace &W, const void *h, int T,
                           const int32_t *idx, const float *gate, float *out, int mode,
                           const uint8_t *one_part, int nparts, cudaStream_t s);
// Tokens per chunk of the grouped tensor-core path.
constexpr int kGroupTokens = 128;
// Default tokens an expert needs in one call to take the tensor-core path.
constexpr int kDefaultMmaMinTokens = 4;
// Batched forward: slots grouped by expert; experts with at least min_tokens tokens
// through the tensor-core kernels, the rest through the lookup kernels.
cudaError_t launch_grouped_forward(const LayerView &L, const Workspace &W, const void *h, int T,
                                   const int32_t *idx, const float *gate, float *out, int mode,
                                   int min_tokens, bool reconstruct, int num_sms, cudaStream_t s,
                                   Timing *tm);
// Row blocks of the down matrix per (slot, segment pair) for the lookup kernels.
int down_row_blocks(int slots, int npair, int groups, int num_sms);
// Whether the fused step kernel can run this call (else the per-phase kernels do).
bool fused_eligible(const LayerView &L, int T, bool with_route, int num_sms);
// Route (optional) and forward in one persistent kernel.
cudaError_t launch_fused_step(const LayerView &L, const Workspace &W, const void *h, int T,
                              bool with_route, int32_t *idx, float *gate, float *logits,
                              const int32_t *pred_idx, int32_t *pred_count, int pred_stride,
                              float *out, int mode, bool reconstruct, int num_sms,
                              cudaStream_t s, unsigned long long *trace = nullptr,
                              int trace_cap = 0, const BankLanes *lanes = nullptr,
                              const int32_t *slot_order = nullptr);
cudaError_t launch_prefetch_l2(const LayerView &L, const int32_t *pred_idx, int pred_stride,
                               int T, int P, int32_t *pred_count, unsigned long long *stats,
                               cudaStream_t s);
cudaError_t launch_pack(const MatGeom &gu, const MatGeom &dn, int n_experts,
                        const uint8_t *gate_codes, const uint8_t *up_codes,
                        const uint8_t *down_codes, uint8_t *records, size_t stride,
                        const size_t sec_off[3], cudaStream_t s);

cudaError_t launch_headers(uint8_t *records, size_t stride, int n, const waste_record_header &hdr,
                           int expert_begin, cudaStream_t s);

cudaError_t launch_rmsnorm(const float *in, float *out, int T, int d, cudaStream_t s);

// crc32 (IEEE 802.3 / zlib) of bytes [payload_off, payload_off + payload_bytes) of each of
// n_records records into crc_out[n_records]; payload_bytes a multiple of 4096; scratch of
// crc_scratch_words(payload_bytes, n_records) words.
cudaError_t launch_payload_crc(const uint8_t *records, size_t stride, int n_records, size_t payload_off,
                               size_t payload_bytes, uint32_t *scratch, uint32_t *crc_out, int num_sms,
                               cudaStream_t s);
size_t crc_scratch_words(size_t payload_bytes, int n_records);
// crc[i] into the 32-bit field at field_off of record i.
cudaError_t launch_crc_store(const uint32_t *crc, uint8_t *records, size_t stride, int n_records,
                             size_t field_off, cudaStream_t s);

int device_sm_count();

// Tiered bank: bring the experts ids[0..n_ids) of `layer` into the HBM cache (demand: the
// clock advances and hits / misses are counted; lookahead: slots of the call in flight stay).
cudaError_t launch_bank_fetch(waste_bank *b, int layer, const int32_t *ids, int n_ids, bool demand,
                              cudaStream_t s);
// A demand fetch whose copy runs inside the persistent step kernel: the plan alone (after the
// bank's last lookahead), which also writes for each of the n_ids slots the job its record
// arrives by (wait_job, -1: resident) and an order of the slots -- resident ones first, then
// by job -- for the units (order).  n_ids <= kOverlapMaxSlots.  The caller then launches the
// step kernel with *lanes on the same stream.
constexpr int kOverlapMaxSlots = 64;
cudaError_t launch_bank_plan_overlap(waste_bank *b, int layer, const int32_t *ids, int n_ids, int32_t *wait_job,
                                     int32_t *order, BankLanes *lanes, cudaStream_t s);
const uint8_t *bank_host_records(const waste_bank *b, int layer);
const uint8_t *bank_slots(const waste_bank *b);
const int32_t *bank_slot_map(const waste_bank *b, int layer);
int bank_layers(const waste_bank *b);
int bank_slot_count(const waste_bank *b);
size_t bank_stride(const waste_bank *b);
const waste_moe_config &bank_config(const waste_bank *b);
// Predicted-expert count of each token (the lookahead's P), read by the next route.
cudaError_t launch_set_pred_count(int32_t *pred_count, int T, int P, cudaStream_t s);


// Sets the calling thread's message returned by waste_moe_last_error().
void set_last_error(const char *msg);

// A range named after a C-ABI call on the profiler's timeline for the call's duration (NVTX;
// nothing is recorded unless a profiler is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

} // namespace wm
