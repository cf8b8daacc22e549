// Tiered expert bank: the records of several layers in host memory (pinned, read by the
// GPU over the CPU-GPU link), an HBM cache of n_slots records, and the device-side fetch
// that brings a call's experts into the cache.
//
// Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", sections "Budget RAM et zone
// de performance étroite" and "Lecture anticipée et prédiction du routeur": the trunk stays
// resident, a bounded cache holds experts, a miss reads the expert's record from the slow
// tier, and a lookahead on the next layer's router fills the cache ahead of demand (their
// demand hit rate rises from 14% to 38% with the bytes read unchanged).  Here the slow tier
// is Grace memory and the fast one HBM.
//
// A fetch is two kernels on the caller's stream: a plan (one warp: first every requested
// expert already resident takes the call's stamp; then each miss takes the least recently
// used slot whose tick is older than the current clock -- slots stamped by the call in flight
// are never victims -- and becomes a copy job) and a copy (a few CTAs, which keep the link
// busy while leaving the SMs to the expert kernels).  A demand fetch of a decode call can
// instead leave the copy to the persistent step kernel, which consumes each expert as its
// copy lands (launch_bank_plan_overlap).  The expert -> slot map is what the expert kernels
// read through.  Fetches must not overlap: the caller orders them (one stream, or events
// between streams).
#include <new>

#include "bank_dev.cuh"

struct waste_bank {
    waste_moe_config cfg;
    int n_layers, E, n_slots;
    size_t stride;
    const uint8_t *host;  // device-usable address of the host records
    wm::BankDevice D;
    // the last demand fetch (for a fetch whose copy runs in the step kernel: its plan) and the
    // last lookahead fetch: each kind waits for the other, so plans never overlap and a
    // lookahead copies only into slots no running expert kernel reads, whatever streams the
    // fetches are issued on
    cudaEvent_t ev_demand, ev_lookahead;
    int2 *jobs[2];       // copy jobs of the last plan of each kind (demand, lookahead)
    int32_t *n_jobs[2];
};

namespace wm {

namespace {

// The bank's device state with the job list of one kind of fetch (a lookahead may plan and
// copy while the step kernel of a demand fetch still reads its own jobs).
BankDevice device_for(const waste_bank *b, bool demand) {
    BankDevice D = b->D;
    D.jobs = b->jobs[demand ? 0 : 1];
    D.n_jobs = b->n_jobs[demand ? 0 : 1];
    return D;
}

// Ranks of positions by (wait_job, position), resident ones (-1) first: order[rank] = position.
__device__ __forceinline__ void plan_order(const int32_t *wait_job, int32_t *order, int n_ids, int lane) {
    for (int p = lane; p < n_ids; p += 32) {
        const int kp = wait_job[p];
        int r = 0;
        for (int q = 0; q < n_ids; ++q) {
            const int kq = wait_job[q];
            r += (kq < kp) || (kq == kp && q < p);
        }
        order[r] = p;
    }
}

// One warp; the slots' ticks and keys in shared memory (2 x n_slots words).  With wait_job /
// order (n_ids <= 64): wait_job[i] = the job by which id i's record arrives in this fetch, or -1
// when it is already resident (or has no slot); order = the ids' positions sorted by (wait_job,
// position), resident ones first.
//  1. every requested expert already resident takes this call's stamp (no miss evicts it);
//  2. the ids in order, 32 at a time with their slots loaded together: a resident one is a hit;
//     a miss takes the least (tick, index) slot older than the call -- each lane keeps the least
//     of its own slots (v = lane mod 32), so a miss is a warp minimum and one lane's rescan --
//     and becomes a job; a later id of the same expert sees the placement (a hit on that job).
__global__ void __launch_bounds__(32) plan_kernel(BankDevice D, int layer, int E, int n_slots, size_t stride,
                                                  const int32_t *__restrict__ ids, int n_ids, int demand,
                                                  int32_t *__restrict__ wait_job, int32_t *__restrict__ order) {
    extern __shared__ uint32_t plan_smem[];
    uint32_t *tick = plan_smem;                                   // [n_slots]
    int32_t *key_of = reinterpret_cast<int32_t *>(plan_smem + n_slots); // [n_slots]
    const int lane = threadIdx.x;
    uint32_t clock = *D.clock;
    if (demand) clock += 1;
    const uint32_t seq = *D.seq + 1;
    // the first 32 ids and their slots, loaded beside the slot state
    int key0 = -1, slot0 = -1;
    const int e0 = lane < n_ids ? ids[lane] : -1;
    for (int v = lane; v < n_slots; v += 32) {
        tick[v] = D.tick[v];
        key_of[v] = D.key_of[v];
    }
    if (e0 >= 0 && e0 < E) {
        key0 = layer * E + e0;
        slot0 = D.map[key0];
    }
    __syncwarp();
    if (lane == 0) {
        *D.clock = clock;
        *D.seq = seq;
    }
    if (slot0 >= 0) {
        tick[slot0] = clock;
        D.tick[slot0] = clock;
    }
    for (int i = 32 + lane; i < n_ids; i += 32) {
        const int e = ids[i];
        if (e < 0 || e >= E) continue;
        const int s = D.map[layer * E + e];
        if (s >= 0) {
            tick[s] = clock;
            D.tick[s] = clock;
        }
    }
    __syncwarp();
    // this lane's least (tick, index) among its slots older than the call
    auto lane_min = [&]() {
        unsigned long long best = ~0ull;
        for (int v = lane; v < n_slots; v += 32) {
            const uint32_t t = tick[v];
            if (t < clock) {
                const unsigned long long c = ((unsigned long long)t << 32) | (unsigned)v;
                best = c < best ? c : best;
            }
        }
        return best;
    };
    unsigned long long mine = lane_min();
    int n_jobs = 0;
    unsigned long long hits = 0, misses = 0;
    for (int i0 = 0; i0 < n_ids; i0 += 32) {
        const int i = i0 + lane;
        int key = key0, slot = slot0, wj = -1;
        if (i0 > 0) {
            key = -1;
            slot = -1;
            if (i < n_ids) {
                const int e = ids[i];
                if (e >= 0 && e < E) {
                    key = layer * E + e;
                    slot = D.map[key];
                    // placed by an earlier chunk of this plan: waits for that job
                    if (slot >= 0 && D.job_seq[slot] == seq) wj = D.job_of[slot];
                }
            }
        }
        const int n = min(32, n_ids - i0);
        for (int j = 0; j < n; ++j) {
            const int kj = __shfl_sync(0xffffffffu, key, j);
            const int sj = __shfl_sync(0xffffffffu, slot, j);
            if (kj < 0) continue;
            if (sj >= 0) {
                ++hits;
                continue;
            }
            unsigned long long best = mine;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const unsigned long long b = __shfl_xor_sync(0xffffffffu, best, o);
                best = b < best ? b : best;
            }
            if (best == ~0ull) continue; // every slot is in use by this call: left unplaced
            const int v = (int)(best & 0xffffffffu);
            if (lane == 0) {
                const int old = key_of[v];
                if (old >= 0) D.map[old] = -1;
                D.map[kj] = v;
                D.key_of[v] = kj;
                D.tick[v] = clock;
                D.jobs[n_jobs] = make_int2(v, kj);
                D.job_seq[v] = seq;
                D.job_of[v] = n_jobs;
                key_of[v] = kj;
                tick[v] = clock;
            }
            __syncwarp();
            if ((v & 31) == lane) mine = lane_min(); // the owner of slot v looks again
            if (key == kj) { // this id and every later one of the same expert: on this job
                slot = v;
                wj = n_jobs;
            }
            ++n_jobs;
            ++misses;
        }
        if (wait_job && i < n_ids) wait_job[i] = wj;
    }
    if (order) {
        __syncwarp();
        plan_order(wait_job, order, n_ids, lane);
    }
    if (lane == 0) { // reductions, so the warp does not wait for the counters' old values
        *D.n_jobs = n_jobs;
        atomicAdd(D.stats + (demand ? kBankDemandHits : kBankPrefetchPresent), hits);
        atomicAdd(D.stats + (demand ? kBankDemandMisses : kBankPrefetchCopies), misses);
        atomicAdd(D.stats + kBankCopiedBytes, (unsigned long long)n_jobs * stride);
    }
}

// The plan with the slot state read from global memory, for banks whose ticks and keys do not
// fit in shared memory (same decisions as plan_kernel).
__global__ void __launch_bounds__(32) plan_kernel_global(BankDevice D, int layer, int E, int n_slots, size_t stride,
                                                  const int32_t *__restrict__ ids, int n_ids, int demand,
                                                  int32_t *__restrict__ wait_job, int32_t *__restrict__ order) {
    const int lane = threadIdx.x;
    uint32_t clock = *D.clock;
    if (demand) clock += 1;
    const uint32_t seq = *D.seq + 1;
    __syncwarp();
    if (lane == 0) {
        *D.clock = clock;
        *D.seq = seq;
    }
    // first every requested expert already resident takes this call's stamp, so that no miss
    // below can evict it
    for (int i = lane; i < n_ids; i += 32) {
        const int e = ids[i];
        if (e < 0 || e >= E) continue;
        const int s = D.map[layer * E + e];
        if (s >= 0) D.tick[s] = clock;
    }
    __syncwarp();
    int n_jobs = 0;
    unsigned long long hits = 0, misses = 0;
    for (int i = 0; i < n_ids; ++i) {
        const int e = ids[i];
        if (e < 0 || e >= E) {
            if (wait_job && lane == 0) wait_job[i] = -1;
            continue;
        }
        const int key = layer * E + e;
        const int s = D.map[key];
        __syncwarp();
        if (s >= 0) {
            if (lane == 0) {
                D.tick[s] = clock;
                // a repeat of an expert this plan is copying waits for the same job
                if (wait_job) wait_job[i] = D.job_seq[s] == seq ? D.job_of[s] : -1;
            }
            ++hits;
            __syncwarp();
            continue;
        }
        // least recently used slot older than this call: (tick, index) minimum over the warp
        unsigned long long best = ~0ull;
        for (int v = lane; v < n_slots; v += 32) {
            const uint32_t t = D.tick[v];
            if (t < clock) {
                const unsigned long long c = ((unsigned long long)t << 32) | (unsigned)v;
                best = c < best ? c : best;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const unsigned long long b = __shfl_xor_sync(0xffffffffu, best, o);
            best = b < best ? b : best;
        }
        if (best == ~0ull) { // every slot is in use by this call: left unplaced
            if (wait_job && lane == 0) wait_job[i] = -1;
            continue;
        }
        const int v = (int)(best & 0xffffffffu);
        if (lane == 0) {
            const int old = D.key_of[v];
            if (old >= 0) D.map[old] = -1;
            D.map[key] = v;
            D.key_of[v] = key;
            D.tick[v] = clock;
            D.jobs[n_jobs] = make_int2(v, key);
            D.job_seq[v] = seq;
            D.job_of[v] = n_jobs;
            if (wait_job) wait_job[i] = n_jobs;
        }
        ++n_jobs;
        ++misses;
        __syncwarp();
    }
    if (order) {
        __syncwarp();
        plan_order(wait_job, order, n_ids, lane);
    }
    if (lane == 0) { // reductions, so the warp does not wait for the counters' old values
        *D.n_jobs = n_jobs;
        atomicAdd(D.stats + (demand ? kBankDemandHits : kBankPrefetchPresent), hits);
        atomicAdd(D.stats + (demand ? kBankDemandMisses : kBankPrefetchCopies), misses);
        atomicAdd(D.stats + kBankCopiedBytes, (unsigned long long)n_jobs * stride);
    }
}

__global__ void __launch_bounds__(bank::kCopyThreads) copy_kernel(BankDevice D, const uint8_t *__restrict__ host,
                                                                  size_t stride) {
    bank::copy_jobs(D, host, stride, *D.n_jobs, (int)blockIdx.x, (int)gridDim.x, [](int) {});
}

} // namespace

// The plan: with the slots' ticks and keys in shared memory when they fit in 48 KiB, else
// read from global memory (same decisions).
void launch_plan(const waste_bank *b, const BankDevice &D, int layer, const int32_t *ids, int n_ids, bool demand,
                 int32_t *wait_job, int32_t *order, cudaStream_t s) {
    const size_t smem = (size_t)b->n_slots * 8;
    if (smem <= 48 * 1024)
        plan_kernel<<<1, 32, smem, s>>>(D, layer, b->E, b->n_slots, b->stride, ids, n_ids, demand ? 1 : 0, wait_job,
                                        order);
    else
        plan_kernel_global<<<1, 32, 0, s>>>(D, layer, b->E, b->n_slots, b->stride, ids, n_ids, demand ? 1 : 0,
                                            wait_job, order);
}

cudaError_t launch_bank_fetch(waste_bank *b, int layer, const int32_t *ids, int n_ids, bool demand,
                              cudaStream_t s) {
    cudaError_t e = cudaStreamWaitEvent(s, demand ? b->ev_lookahead : b->ev_demand, 0);
    if (e != cudaSuccess) return e;
    const BankDevice D = device_for(b, demand);
    launch_plan(b, D, layer, ids, n_ids, demand, nullptr, nullptr, s);
    copy_kernel<<<bank::kCopyLanes, bank::kCopyThreads, 0, s>>>(D, b->host, b->stride);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return cudaEventRecord(demand ? b->ev_demand : b->ev_lookahead, s);
}

cudaError_t launch_bank_plan_overlap(waste_bank *b, int layer, const int32_t *ids, int n_ids, int32_t *wait_job,
                                     int32_t *order, BankLanes *lanes, cudaStream_t s) {
    if (n_ids > kOverlapMaxSlots) return cudaErrorInvalidValue;
    cudaError_t e = cudaStreamWaitEvent(s, b->ev_lookahead, 0);
    if (e != cudaSuccess) return e;
    const BankDevice D = device_for(b, true);
    launch_plan(b, D, layer, ids, n_ids, true, wait_job, order, s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    lanes->D = D;
    lanes->host = b->host;
    lanes->wait_job = wait_job;
    lanes->lanes = bank::kCopyLanes;
    // a lookahead into the next layer may plan from here on: it evicts no slot of this call
    return cudaEventRecord(b->ev_demand, s);
}

const uint8_t *bank_host_records(const waste_bank *b, int layer) {
    return b->host + (size_t)layer * b->E * b->stride;
}
const uint8_t *bank_slots(const waste_bank *b) { return b->D.slots; }
const int32_t *bank_slot_map(const waste_bank *b, int layer) { return b->D.map + (size_t)layer * b->E; }
int bank_layers(const waste_bank *b) { return b->n_layers; }
int bank_slot_count(const waste_bank *b) { return b->n_slots; }
size_t bank_stride(const waste_bank *b) { return b->stride; }
const waste_moe_config &bank_config(const waste_bank *b) { return b->cfg; }

} // namespace wm

using namespace wm;

namespace {
int bank_fail(int code, const char *msg) {
    set_last_error(msg);
    return code;
}
} // namespace

extern "C" {

int waste_bank_create(const waste_moe_config *cfg, int32_t n_layers, const uint8_t *host_records,
                      size_t record_stride, int32_t n_slots, waste_bank **out) {
    const NvtxRange nvtx_range(__func__);
    if (!out) return bank_fail(WASTE_EINVAL, "out is NULL");
    *out = nullptr;
    size_t min_stride = 0;
    int rc = waste_moe_record_layout(cfg, &min_stride, nullptr, nullptr);
    if (rc) return rc;
    if (n_layers < 1 || n_slots < 1 || !host_records)
        return bank_fail(WASTE_EINVAL, "n_layers and n_slots must be >= 1, host_records not NULL");
    if (record_stride < min_stride || record_stride % WASTE_RECORD_ALIGN)
        return bank_fail(WASTE_ELAYOUT, "record stride too small or not a multiple of 4096");
    if ((size_t)n_layers * cfg->n_experts > 0x7fffffff)
        return bank_fail(WASTE_EINVAL, "too many records");
    void *dev = nullptr;
    cudaError_t e = cudaHostGetDevicePointer(&dev, const_cast<uint8_t *>(host_records), 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return bank_fail(WASTE_EINVAL, "host_records is not host memory the device can read");
    }
    if (((uintptr_t)dev) % WASTE_RECORD_ALIGN || ((uintptr_t)host_records) % WASTE_RECORD_ALIGN)
        return bank_fail(WASTE_ELAYOUT, "host_records must be 4096-aligned");
    waste_bank *b = new (std::nothrow) waste_bank();
    if (!b) return bank_fail(WASTE_ENOMEM, "host allocation");
    b->cfg = *cfg;
    b->n_layers = n_layers;
    b->E = cfg->n_experts;
    b->n_slots = n_slots;
    b->stride = record_stride;
    b->host = static_cast<const uint8_t *>(dev);
    const size_t keys = (size_t)n_layers * b->E;
    const size_t slot_bytes = (size_t)n_slots * record_stride;
    const size_t meta = keys * 4 + (size_t)n_slots * (4 + 4 + 8 + 8 + 4 + 4) + 256 + kBankStatCount * 8;
    void *mem = nullptr;
    e = cudaMalloc(&mem, slot_bytes + round_up(meta, 256) + 256);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete b;
        return bank_fail(WASTE_ENOMEM, "HBM cache allocation");
    }
    uint8_t *p = static_cast<uint8_t *>(mem);
    b->D.base = mem;
    b->D.slots = p;
    p += slot_bytes;
    b->D.map = reinterpret_cast<int32_t *>(p);
    p += round_up(keys * 4, 16);
    b->D.key_of = reinterpret_cast<int32_t *>(p);
    p += round_up((size_t)n_slots * 4, 16);
    b->D.tick = reinterpret_cast<uint32_t *>(p);
    p += round_up((size_t)n_slots * 4, 16);
    b->jobs[0] = reinterpret_cast<int2 *>(p);
    p += round_up((size_t)n_slots * 8, 16);
    b->jobs[1] = reinterpret_cast<int2 *>(p);
    p += round_up((size_t)n_slots * 8, 16);
    b->D.jobs = b->jobs[0];
    b->D.job_seq = reinterpret_cast<uint32_t *>(p);
    p += round_up((size_t)n_slots * 4, 16);
    b->D.job_of = reinterpret_cast<int32_t *>(p);
    p += round_up((size_t)n_slots * 4, 16);
    b->D.clock = reinterpret_cast<uint32_t *>(p);
    b->n_jobs[0] = reinterpret_cast<int32_t *>(p + 4);
    b->D.seq = reinterpret_cast<uint32_t *>(p + 8);
    b->n_jobs[1] = reinterpret_cast<int32_t *>(p + 12);
    b->D.n_jobs = b->n_jobs[0];
    p += 16;
    b->D.stats = reinterpret_cast<unsigned long long *>(p);
    b->ev_demand = b->ev_lookahead = nullptr;
    e = cudaEventCreateWithFlags(&b->ev_demand, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b->ev_lookahead, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        cudaGetLastError();
        waste_bank_destroy(b);
        return bank_fail(WASTE_ECUDA, "bank events");
    }
    *out = b;
    rc = waste_bank_reset(b);
    if (rc) {
        waste_bank_destroy(b);
        *out = nullptr;
    }
    return rc;
}

void waste_bank_destroy(waste_bank *b) {
    if (!b) return;
    cudaDeviceSynchronize();
    if (b->ev_demand) cudaEventDestroy(b->ev_demand);
    if (b->ev_lookahead) cudaEventDestroy(b->ev_lookahead);
    cudaFree(b->D.base);
    delete b;
}

int waste_bank_reset(waste_bank *b) {
    if (!b) return bank_fail(WASTE_EINVAL, "NULL bank");
    const size_t keys = (size_t)b->n_layers * b->E;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemset(b->D.map, 0xff, keys * 4);
    if (e == cudaSuccess) e = cudaMemset(b->D.key_of, 0xff, (size_t)b->n_slots * 4);
    if (e == cudaSuccess) e = cudaMemset(b->D.tick, 0, (size_t)b->n_slots * 4);
    if (e == cudaSuccess) e = cudaMemset(b->D.job_seq, 0, (size_t)b->n_slots * 4);
    if (e == cudaSuccess) e = cudaMemset(b->D.clock, 0, 16);
    if (e == cudaSuccess) e = cudaMemset(b->D.stats, 0, kBankStatCount * 8);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return bank_fail(WASTE_ECUDA, cudaGetErrorString(e));
    set_last_error("");
    return WASTE_OK;
}

int waste_bank_stats(const waste_bank *b, waste_bank_stats_t *out) {
    if (!b || !out) return bank_fail(WASTE_EINVAL, "NULL bank or output");
    unsigned long long v[kBankStatCount];
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(v, b->D.stats, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return bank_fail(WASTE_ECUDA, cudaGetErrorString(e));
    out->demand_hits = v[kBankDemandHits];
    out->demand_misses = v[kBankDemandMisses];
    out->prefetch_copies = v[kBankPrefetchCopies];
    out->prefetch_present = v[kBankPrefetchPresent];
    out->copied_bytes = v[kBankCopiedBytes];
    set_last_error("");
    return WASTE_OK;
}

} // extern "C"
