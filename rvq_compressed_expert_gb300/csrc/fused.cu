// One persistent kernel for a whole decode step of one MoE layer: router GEMV,
// top-k + softmax, the table-lookup gate/up units, the down units and the
// gate-weighted combine, in one launch.
//
// Work items are claimed from a device-side queue in a fixed order:
//   [router items][top-k item][copy lanes][gate/up units][down units][combine items]
// Copy lanes exist for a call on a tiered bank whose demand copies run in this kernel
// (page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée et
// prédiction du routeur": each of a layer's expert reads is issued on its own and the
// compute consumes each expert as it arrives, with the work and cache statistics unchanged).  The lanes copy the missing records job by job, chunk by chunk,
// and count the chunks of each job; the units of a slot whose record is on its way wait for
// its count, while the units of resident experts -- ordered first -- run beside the copy.
// A copy lane does not claim its next item before it finishes, so it holds no unit back.
// A CTA claims one item ahead of the one it runs, so the next unit's codes and
// codebooks can be fetched while the current one streams.  An item waits only on
// items that precede it in the queue (top-k on all router items, gate/up units on
// the top-k, a down unit on the gate/up units of its slot, a combine item on the
// down units of its rows), signalled by device counters with release/acquire
// ordering.  Because every CTA runs its items in claim order, the smallest
// unfinished item never waits on anything unfinished, so the queue always makes
// progress whatever number of CTAs is resident; every wait is still bounded and
// records kErrTimeout if it gives up.  The last CTA to leave resets the counters
// for the next launch.  The arithmetic of each item is that of the per-phase
// kernels, in the same order: results are bit-identical to them.
#include <cstring>

#include "bank_dev.cuh"
#include "lut_dev.cuh"
#include "route_dev.cuh"

namespace wm {

using namespace lut;
using namespace route;

namespace {

constexpr int kRouterRowsPerItem = kThreads / 128; // 4 expert rows per router item
constexpr int kCombineRows = kThreads;              // output rows per combine item
constexpr int kMaxFusedExperts = 1024;              // top-k of the step kernel sorts <= 1024 keys
static_assert(kThreads == bank::kCopyThreads, "a copy lane is one CTA of the step kernel");
// L2 prefetch distance of the step kernel's units, which load a whole round of codes at the
// top of each round (three rounds measured best for that order)
constexpr int kStepPrefetchRounds = 3;

struct FusedArgs {
    LutArgs A; // lookup units; A.idx is where the top-k item writes the routing
    // routing
    const float *router_w, *router_b;
    float *logits, *logits_lo; // [T][E]
    int32_t *idx_out;
    float *gate_out;
    const int32_t *pred_idx;
    int32_t *pred_count;
    int pred_stride;
    unsigned long long router_bytes;
    int with_route;
    int T, d;
    // combine
    const float *gate, *h32;
    float *out;
    int mode;
    // queue and counters (zero at rest):
    // [0] next item, [1] CTAs that left, [2] router items done, [3] top-k done,
    // [4, 4 + slots) gate/up units done per slot, then down units done per row block, then
    // chunks copied per copy job (banked calls)
    unsigned *sync;
    int n_router, n_topk, n_copy, n_gu, n_dn, n_comb;
    BankLanes bank;          // n_copy > 0 only
    int bank_copiers;        // copy lanes that count themselves on each job
    // optional item trace: per item {start ns, end ns, SM id, CTA} (null = off)
    unsigned long long *trace;
    int trace_cap;
};

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned smid() {
    unsigned r;
    asm volatile("mov.u32 %0, %smid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void signal(unsigned *c) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(c, 1u);
    }
}

__device__ __forceinline__ int claim(unsigned *q, int *slot) {
    __syncthreads();
    if (threadIdx.x == 0) *slot = (int)atomicAdd(q, 1u);
    __syncthreads();
    return *slot;
}

// The cold items run out of line, so their registers do not add to the units'.
template <bool kBf16>
__device__ __noinline__ void router_item(const FusedArgs &F, int item, float (*red)[4][kRouterTok]) {
    // hidden states staged in the (idle) table area of shared memory
    const int hs_tokens = (int)min((size_t)kRouterTok, (size_t)kTabBytes / ((size_t)F.d * 4));
    router_block_staged<kBf16>(F.router_w, F.router_b, F.A.h, F.T, F.A.E, F.d,
                               item * kRouterRowsPerItem, F.logits, F.logits_lo, red,
                               reinterpret_cast<float *>(lut_smem), hs_tokens);
}

__device__ __noinline__ void topk_item(const FusedArgs &F) {
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(lut_smem);
    int *ids = reinterpret_cast<int *>(lut_smem + 8 * kMaxFusedExperts);
    for (int t = 0; t < F.T; ++t)
        topk_block(F.logits, F.logits_lo, F.A.E, F.A.k, t, F.idx_out, F.gate_out, F.pred_idx,
                   F.pred_count, F.pred_stride, F.A.stats, F.router_bytes, keys, ids);
}

// combine rows [r0, r1) of every token from the down partials (same order as the
// per-phase combine kernel)
__device__ __noinline__ void combine_item(const FusedArgs &F, int r0, int r1) {
    // kernel parameters copied to registers once (read through a reference inside the
    // loops they would be local-memory loads)
    const int d = F.d, k = F.A.k, T = F.T, mode = F.mode, E = F.A.E, npair = F.A.npair;
    const int32_t *__restrict__ idx = F.A.idx;
    const float *__restrict__ gate = F.gate;
    const float *__restrict__ part_dn = F.A.part_dn;
    const float *__restrict__ h32 = F.h32;
    float *__restrict__ out = F.out;
    for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        for (int t = 0; t < T; ++t) {
            float y = 0.f;
            for (int i0 = 0; i0 < k; i0 += 8) {
                float sv[8], gv[8];
                bool ok[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    // loads of 8 slots go out together: slots past k are clamped to the last
                    // one and masked
                    const int i = min(i0 + u, k - 1);
                    const int e = idx[(size_t)t * k + i];
                    ok[u] = (i0 + u < k) && e >= 0 && e < E;
                    gv[u] = gate[(size_t)t * k + i];
                    const float *p = part_dn + ((size_t)t * k + i) * npair * d + r;
                    float s = 0.f;
#pragma unroll 4
                    for (int q = 0; q < npair; ++q) s += p[(size_t)q * d];
                    sv[u] = s;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (ok[u]) y = fmaf(gv[u], sv[u], y);
            }
            const size_t o = (size_t)t * d + r;
            if (mode == 0) out[o] = y;
            else if (mode == 1) out[o] = out[o] + y;
            else out[o] = h32[o] + y;
        }
    }
}

// Queue layout helpers: item boundaries and counters are recomputed from the
// kernel parameters where needed, so little state stays live across a unit.
__device__ __forceinline__ int b_topk(const FusedArgs &F) { return F.n_router; }
__device__ __forceinline__ int b_copy(const FusedArgs &F) { return F.n_router + F.n_topk; }
__device__ __forceinline__ int b_gu(const FusedArgs &F) { return b_copy(F) + F.n_copy; }
__device__ __forceinline__ int b_dn(const FusedArgs &F) { return b_gu(F) + F.n_gu; }
__device__ __forceinline__ int b_comb(const FusedArgs &F) { return b_dn(F) + F.n_dn; }
__device__ __forceinline__ int n_total(const FusedArgs &F) { return b_comb(F) + F.n_comb; }
__device__ __forceinline__ unsigned *gu_done(const FusedArgs &F) { return F.sync + 4; }
__device__ __forceinline__ unsigned *dn_done(const FusedArgs &F) { return F.sync + 4 + F.A.slots; }
__device__ __forceinline__ unsigned *job_done(const FusedArgs &F) { return F.sync + 4 + F.A.slots + F.A.nrb; }
template <bool kBanked>
__device__ __forceinline__ bool is_copy(const FusedArgs &F, int item) {
    return kBanked && item >= b_copy(F) && item < b_gu(F);
}

// Copy lane `lane`: chunks lane, lane + n_copy, ... of the plan's jobs, so the lanes finish
// the jobs in order; a lane counts itself on a job after its last chunk of the job.
__device__ __noinline__ void copy_item(const FusedArgs &F, int lane) {
    unsigned *done = job_done(F);
    bank::copy_jobs(F.bank.D, F.bank.host, F.A.stride, *F.bank.D.n_jobs, lane, F.n_copy,
                    [&](int j) { signal(done + j); });
}

// Before any code of `slot` is read: wait until its record, if it is being copied, is in.
template <bool kBanked>
__device__ __forceinline__ void wait_record(const FusedArgs &F, int slot) {
    if (kBanked) {
        const int j = F.bank.wait_job[slot];
        if (j >= 0) wait_counter(job_done(F) + j, (unsigned)F.bank_copiers, F.A.err);
    }
}

// kBanked: a call on a tiered bank with copy lanes (its own instance, so the copy code adds
// nothing to the registers of the resident-record instances)
template <bool kRecon, bool kBf16, bool kBanked>
__global__ void __launch_bounds__(kThreads, 1) fused_step_kernel(const FusedArgs F) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float red[kRouterRowsPerItem][4][kRouterTok];
    __shared__ int claimed;
    bool primed = false;
    TabTc tcs;
    tab_tc_open<kRecon>(tcs);
    int cur = claim(F.sync, &claimed);
    int nxt = is_copy<kBanked>(F, cur) ? -1 : claim(F.sync, &claimed);
    while (cur < n_total(F)) {
        unsigned long long t_start = 0;
        if (F.trace && threadIdx.x == 0) t_start = globaltimer();
        if (cur < b_copy(F)) {
            // a banked call is routed before the kernel: its instance has no routing items
            if constexpr (!kBanked) {
                if (cur < b_topk(F)) {
                    // ---- router rows
                    router_item<kBf16>(F, cur, red);
                    signal(F.sync + 2);
                } else {
                    // ---- top-k + softmax of every token, one warp per token
                    wait_counter(F.sync + 2, (unsigned)F.n_router, F.A.err);
                    topk_item(F);
                    __syncthreads();
                    if (threadIdx.x == 0) {
                        __threadfence();
                        atomicExch(F.sync + 3, 1u);
                    }
                }
            }
        } else if (cur < b_gu(F)) {
            // ---- copy lane of a banked call
            if constexpr (kBanked) copy_item(F, cur - b_copy(F));
        } else if (cur < b_dn(F)) {
            // ---- gate/up unit
            if (F.with_route) wait_counter(F.sync + 3, 1u, F.A.err);
            const Unit U = decode_unit<false>(F.A, cur - b_gu(F));
            wait_record<kBanked>(F, U.slot);
            const bool has_next = nxt >= b_gu(F) && nxt < b_dn(F);
            Unit N;
            if (has_next) N = decode_unit<false>(F.A, nxt - b_gu(F));
            run_unit<false, kRecon, kBf16, kThreads, kBanked ? kPrefetchRounds : kStepPrefetchRounds, kBanked>(
                F.A, U, has_next, N, primed, tcs, nullptr, 0);
            signal(gu_done(F) + U.slot);
        } else if (cur < b_comb(F)) {
            // ---- down unit (waits inside for the gate/up units of its slot)
            if (F.with_route) wait_counter(F.sync + 3, 1u, F.A.err);
            const int u = cur - b_dn(F);
            const Unit U = decode_unit<true>(F.A, u);
            wait_record<kBanked>(F, U.slot);
            const bool has_next = nxt >= b_dn(F) && nxt < b_comb(F);
            Unit N;
            if (has_next) N = decode_unit<true>(F.A, nxt - b_dn(F));
            run_unit<true, kRecon, kBf16, kThreads, kBanked ? kPrefetchRounds : kStepPrefetchRounds, kBanked>(
                F.A, U, has_next, N, primed, tcs, gu_done(F) + U.slot, (unsigned)(2 * F.A.gu_pairs));
            signal(dn_done(F) + (u % F.A.nrb));
        } else {
            // ---- combine rows [r0, r1) once every down unit over them is done
            const int r0 = (cur - b_comb(F)) * kCombineRows;
            const int r1 = min(F.d, r0 + kCombineRows);
            const int rb0 = (r0 / kGroupRows) / F.A.rb_groups;
            const int rb1 = ((r1 - 1) / kGroupRows) / F.A.rb_groups;
            for (int rb = rb0; rb <= rb1; ++rb)
                wait_counter(dn_done(F) + rb, (unsigned)(F.A.slots * F.A.npair), F.A.err);
            combine_item(F, r0, r1);
            if (cur == b_comb(F) && threadIdx.x == 0 && F.A.stats)
                atomicAdd(F.A.stats + kStatForwardSlots, (unsigned long long)F.A.slots);
        }
        if (F.trace && threadIdx.x == 0 && cur < F.trace_cap) {
            unsigned long long *e = F.trace + 4 * (size_t)cur;
            e[0] = t_start;
            e[1] = globaltimer();
            e[2] = smid();
            e[3] = blockIdx.x;
        }
        cur = nxt >= 0 ? nxt : claim(F.sync, &claimed);
        nxt = is_copy<kBanked>(F, cur) ? -1 : claim(F.sync, &claimed);
    }

    tab_tc_close<kRecon>(tcs);
    // the last CTA to leave puts the queue and counters back to zero
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned left = atomicAdd(F.sync + 1, 1u);
        if (left == gridDim.x - 1) {
            __threadfence();
            const int n = 4 + F.A.slots + F.A.nrb + (F.n_copy ? F.A.slots : 0);
            for (int i = 0; i < n; ++i) F.sync[i] = 0u;
            __threadfence();
        }
    }
}

template <bool kRecon, bool kBf16, bool kBanked>
cudaError_t launch_fused_t(const FusedArgs &F, int grid, cudaStream_t s) {
    const size_t smem = unit_smem<kRecon>();
    static SmemAttr attr;
    cudaError_t e = ensure_smem(attr, (const void *)fused_step_kernel<kRecon, kBf16, kBanked>, (int)smem);
    if (e != cudaSuccess) return e;
    fused_step_kernel<kRecon, kBf16, kBanked><<<grid, kThreads, smem, s>>>(F);
    return cudaGetLastError();
}

template <bool kRecon, bool kBf16>
cudaError_t launch_fused_b(const FusedArgs &F, int grid, cudaStream_t s) {
    return F.n_copy ? launch_fused_t<kRecon, kBf16, true>(F, grid, s) : launch_fused_t<kRecon, kBf16, false>(F, grid, s);
}

} // namespace

bool fused_eligible(const LayerView &L, int T, bool with_route, int num_sms) {
    const int slots = T * L.k;
    const int npair = (L.dn.nseg + 1) / 2;
    if (down_row_blocks(slots, npair, L.dn.groups, num_sms) > kMaxFusedRowBlocks) return false;
    if (with_route && (L.E > kMaxFusedExperts || (size_t)L.d * 4 > (size_t)kTabBytes)) return false;
    return true;
}

cudaError_t launch_fused_step(const LayerView &L, const Workspace &W, const void *h, int T,
                              bool with_route, int32_t *idx, float *gate, float *logits,
                              const int32_t *pred_idx, int32_t *pred_count, int pred_stride,
                              float *out, int mode, bool reconstruct, int num_sms,
                              cudaStream_t s, unsigned long long *trace, int trace_cap,
                              const BankLanes *lanes, const int32_t *slot_order) {
    FusedArgs F;
    F.trace = trace;
    F.trace_cap = trace_cap;
    LutArgs &A = F.A;
    A.records = L.records;
    A.slot_map = L.slot_map;
    A.stride = L.stride;
    A.codebooks = L.codebooks;
    A.idx = idx;
    A.h = h;
    A.E = L.E;
    A.k = L.k;
    A.slots = T * L.k;
    A.gu = L.gu;
    A.off_gate = L.sec_off[0];
    A.off_up = L.sec_off[1];
    A.gu_pairs = (L.gu.nseg + 1) / 2;
    A.part_gu = W.part_gu;
    A.dn = L.dn;
    A.off_down = L.sec_off[2];
    A.npair = (L.dn.nseg + 1) / 2;
    A.nrb = down_row_blocks(A.slots, A.npair, L.dn.groups, num_sms);
    A.rb_groups = (L.dn.groups + A.nrb - 1) / A.nrb;
    A.part_dn = W.part_dn;
    A.stats = W.stats;
    A.err = W.err;
    A.slot_list = slot_order; // a permutation of the call's slots (the unit counts stay)
    A.n_list = nullptr;
    A.trace = nullptr;
    A.trace_cap = 0;
    A.trace_base = 0;
    F.router_w = L.router_w;
    F.router_b = L.router_b;
    F.logits = logits;
    F.logits_lo = W.logits_lo;
    F.idx_out = idx;
    F.gate_out = gate;
    F.pred_idx = pred_idx;
    F.pred_count = pred_count;
    F.pred_stride = pred_stride;
    F.router_bytes = (unsigned long long)L.E * (unsigned long long)L.d * 4ull;
    F.with_route = with_route ? 1 : 0;
    F.T = T;
    F.d = L.d;
    F.gate = gate;
    F.h32 = reinterpret_cast<const float *>(h);
    F.out = out;
    F.mode = mode;
    F.sync = W.sync;
    F.n_router = with_route ? (L.E + kRouterRowsPerItem - 1) / kRouterRowsPerItem : 0;
    F.n_topk = with_route ? 1 : 0;
    F.n_copy = lanes ? lanes->lanes : 0;
    if (lanes) F.bank = *lanes;
    else memset(&F.bank, 0, sizeof F.bank);
    F.bank_copiers = bank::copiers_per_job(L.stride, F.n_copy);
    F.n_gu = A.slots * 2 * A.gu_pairs;
    F.n_dn = A.slots * A.npair * A.nrb;
    F.n_comb = (L.d + kCombineRows - 1) / kCombineRows;
    const int total = F.n_router + F.n_topk + F.n_copy + F.n_gu + F.n_dn + F.n_comb;
    // a banked call leaves as many SMs as it has copy lanes to the lookahead into the next
    // layer, whose copy kernel then runs beside this one
    const int cap = lanes ? max(1, num_sms - F.n_copy) : num_sms;
    const int grid = total < cap ? total : cap;
    const bool bf16 = L.act_bf16 != 0;
    if (reconstruct) return bf16 ? launch_fused_b<true, true>(F, grid, s) : launch_fused_b<true, false>(F, grid, s);
    return bf16 ? launch_fused_b<false, true>(F, grid, s) : launch_fused_b<false, false>(F, grid, s);
}

} // namespace wm
