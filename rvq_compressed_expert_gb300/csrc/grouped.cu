// Batched decode and prefill: the routed (token, expert) slots of a call grouped by
// expert, and every expert that serves enough tokens applied as a dense product on
// the tensor cores.
//
// Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée et
// prédiction du routeur": one layer of a prefill chunk spans about 550 expert slots, so
// one expert's weights serve many tokens at once.  The weights stay in their 3-stage
// RVQ codes (section "Quantification et exactitude"); here 128-row tiles of codes are
// decoded into tensor memory (the sum of three 256-entry codebook rows per 8-weight
// vector) and fed to tcgen05 MMAs with the expert's tokens as the N side.
//
// Kernels, in launch order:
//   group_kernel   per-expert counts, the slots sorted by expert, the chunk list of the
//                  tensor-core experts (<= 128 tokens each, with their rows in the tiled
//                  activation buffers) and the list of the slots left to the lookup
//                  kernels (experts with fewer than min_tokens tokens)
//   gather_kernel  each chunk's activations as fp16 tiles in the order the MMA reads
//                  them (one contiguous block per K chunk), zero padding included
//   mma_kernel<0>  gate and up of every (chunk, 128-row block): two K passes into two
//                  TMEM accumulators, SwiGLU in the epilogue, written as the fp16 tiles
//                  the down kernel reads
//   mma_kernel<1>  down of every (chunk, 128-row block): y per slot into partial 0
// The lookup kernels serve the listed slots in between, and the combine sums the k
// slots of each token in rank order (one partial for tensor-core slots).
//
// mma_kernel is warp-specialised: one producer warp moves the codes of each 32-vector
// segment of the row block (12 KiB, a bulk copy per row group), another the activation tile
// of each 64-wide K chunk; 16 decode warps turn codes into fp16 weights and store them into
// tensor memory (tcgen05.st), where the MMA reads its A operand; two threads, in two warps,
// issue the MMAs (a chunk of <= 64 tokens: alternate K chunks, into two accumulators the
// epilogue adds; a larger one: half of its tokens each).
// Full/empty mbarriers hand the buffers between them, so decoding, copies and MMAs of
// different chunks overlap.  A CTA takes a contiguous range of items, so an expert's
// codebooks stay in shared memory across its row blocks.
//
// Numerics: codebook rows are rounded to fp16 and summed in fp16 (stage order 0, 1, 2),
// the activations enter as fp16, products accumulate in fp32.  The error is that of
// fp16 operands (relative 2^-11 per operand), which is why the path serves bf16
// activations by default and fp32 ones only when asked.
#include <cuda_fp16.h>

#include "common.cuh"
#include "tc_dev.cuh"

namespace wm {

namespace {

constexpr int kBM = 128;  // output rows per item (MMA M)
constexpr int kBK = 64;   // K per chunk: 8 vectors of 8 weights
constexpr int kKcSeg = 4; // K chunks per 32-vector code segment

// ---------------------------------------------------------------- grouping

constexpr int kGroupThreads = 1024;
constexpr int kExpertsPerThread = kMaxExperts / kGroupThreads; // 4

__device__ __forceinline__ int pad16(int n) { return (n + 15) & ~15; }

// rows the chunks of an expert with c tokens take in the tiled activation buffers
__device__ __forceinline__ int expert_rows(int c) {
    const int full = c / kGroupTokens, rest = c % kGroupTokens;
    return full * kGroupTokens + (rest ? pad16(rest) : 0);
}

__global__ void __launch_bounds__(kGroupThreads) group_kernel(const int32_t *__restrict__ idx, int S,
                                                              int E, int min_tokens, Grouping G) {
    __shared__ int cnt[kMaxExperts];
    __shared__ int cur[kMaxExperts];
    __shared__ int4 wsum[kGroupThreads / 32];
    __shared__ int4 total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kGroupThreads) cnt[e] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += kGroupThreads) {
        const int e = idx[s];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive scans over experts of (slots, tensor-core chunks, tiled rows); the thread
    // owns experts [4 tid, 4 tid + 4)
    int ls[kExpertsPerThread], lc[kExpertsPerThread], lr[kExpertsPerThread];
    int4 mine = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kExpertsPerThread; ++i) {
        const int e = kExpertsPerThread * tid + i;
        const int c = e < E ? cnt[e] : 0;
        const bool tensor = c >= min_tokens && c > 0;
        ls[i] = mine.x;
        lc[i] = mine.y;
        lr[i] = mine.z;
        mine.x += c;
        mine.y += tensor ? (c + kGroupTokens - 1) / kGroupTokens : 0;
        mine.z += tensor ? expert_rows(c) : 0;
    }
    int4 inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, inc.x, o);
        const int b = __shfl_up_sync(0xffffffffu, inc.y, o);
        const int c = __shfl_up_sync(0xffffffffu, inc.z, o);
        if (lane >= o) {
            inc.x += a;
            inc.y += b;
            inc.z += c;
        }
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int4 v = wsum[lane];
        int4 w = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, w.x, o);
            const int b = __shfl_up_sync(0xffffffffu, w.y, o);
            const int c = __shfl_up_sync(0xffffffffu, w.z, o);
            if (lane >= o) {
                w.x += a;
                w.y += b;
                w.z += c;
            }
        }
        wsum[lane] = make_int4(w.x - v.x, w.y - v.y, w.z - v.z, 0);
        if (lane == 31) total = w;
    }
    __syncthreads();
    const int4 ws = wsum[warp];
    const int4 base = make_int4(ws.x + inc.x - mine.x, ws.y + inc.y - mine.y, ws.z + inc.z - mine.z, 0);
#pragma unroll
    for (int i = 0; i < kExpertsPerThread; ++i) {
        const int e = kExpertsPerThread * tid + i;
        if (e >= E) break;
        const int off = base.x + ls[i];
        G.offs[e] = off;
        cur[e] = off;
        const int c = cnt[e];
        if (c >= min_tokens && c > 0) {
            const int nc = (c + kGroupTokens - 1) / kGroupTokens;
            int row = base.z + lr[i];
            for (int j = 0; j < nc; ++j) {
                const int n = min(kGroupTokens, c - j * kGroupTokens);
                G.chunks[base.y + lc[i] + j] = make_int4(e, off + j * kGroupTokens, n, row);
                row += pad16(n);
            }
        }
    }
    if (tid == 0) {
        G.offs[E] = total.x;
        G.counts[0] = total.y;
    }
    __syncthreads();
    // placement in slot order (one warp), and the list of the lookup slots
    if (warp == 0) {
        const unsigned lt = (1u << lane) - 1u;
        int n_lut = 0;
        for (int b = 0; b < S; b += 32) {
            const int s = b + lane;
            const int e = s < S ? idx[s] : -1;
            const bool valid = s < S && e >= 0 && e < E;
            const bool tensor = valid && cnt[e] >= min_tokens;
            const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
            int pos = 0;
            if (valid) pos = cur[e] + __popc(peers & lt);
            __syncwarp();
            if (valid) {
                G.sorted[pos] = s;
                if ((peers & lt) == 0) cur[e] += __popc(peers);
            }
            const unsigned lut = __ballot_sync(0xffffffffu, s < S && !tensor);
            if (s < S) {
                if (!tensor) G.lut_slots[n_lut + __popc(lut & lt)] = s;
                G.one_part[s] = tensor ? 1 : 0;
            }
            n_lut += __popc(lut);
            __syncwarp();
        }
        if (lane == 0) G.counts[1] = n_lut;
    }
}

// Tiled fp16 activations of every chunk: for K chunk kc the npad x 64 tile is one
// contiguous block of npad * 128 bytes made of 8x8 core matrices (token n, 8 inputs ki):
// byte (n >> 3) * 1024 + ki * 128 + (n & 7) * 16.  xg holds the hidden states (gate/up
// input); in ag (down input, written by the gate/up epilogue) the pieces the epilogue
// never writes -- padding tokens, inputs past f -- are zeroed here.
__device__ __forceinline__ uint32_t tile_off(int kc, int npad, int n, int col) {
    return (uint32_t)kc * npad * 128 + (n >> 3) * 1024 + ((col & 63) >> 3) * 128 + (n & 7) * 16;
}

template <bool kBf16>
__global__ void __launch_bounds__(256) gather_kernel(const void *__restrict__ h, Grouping G, int d, int f, int k) {
    const int n_chunks = G.counts[0];
    const int kcd = (d + kBK - 1) / kBK, kcf = (f + kBK - 1) / kBK;
    for (int c = blockIdx.x; c < n_chunks; c += gridDim.x) {
        const int4 ch = G.chunks[c];
        const int start = ch.y, nt = ch.z, rb = ch.w, npad = pad16(nt);
        uint4 *xg = reinterpret_cast<uint4 *>(G.xg + (size_t)rb * kcd * 128);
        const int per_tile = npad * 8;
        for (int p = threadIdx.x; p < kcd * per_tile; p += blockDim.x) {
            const int kc = p / per_tile, o = p - kc * per_tile;
            const int n = ((o >> 6) << 3) | (o & 7), ki = (o >> 3) & 7;
            const int col = kc * kBK + ki * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (n < nt && col < d) {
                const int t = G.sorted[start + n] / k;
                float x[8];
                if constexpr (kBf16) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(h) +
                                                                       (size_t)t * d + col);
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
                        x[2 * j] = f2.x;
                        x[2 * j + 1] = f2.y;
                    }
                } else {
                    const float4 a = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(h) +
                                                                       (size_t)t * d + col);
                    const float4 b = *(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(h) +
                                                                        (size_t)t * d + col) + 1);
                    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
                }
                uint32_t *vw = &v.x;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 p2 = __floats2half2_rn(x[2 * j], x[2 * j + 1]);
                    vw[j] = *reinterpret_cast<const uint32_t *>(&p2);
                }
            }
            xg[p] = v;
        }
        uint4 *ag = reinterpret_cast<uint4 *>(G.ag + (size_t)rb * kcf * 128);
        for (int p = threadIdx.x; p < kcf * per_tile; p += blockDim.x) {
            const int kc = p / per_tile, o = p - kc * per_tile;
            const int n = ((o >> 6) << 3) | (o & 7), ki = (o >> 3) & 7;
            if (n >= nt || kc * kBK + ki * 8 >= f) ag[p] = make_uint4(0, 0, 0, 0);
        }
    }
}

// ---------------------------------------------------------------- tensor-core kernels

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
// producers: one warp for the code segments, one for the activation tiles, so neither ring's
// progress holds the other's copies back
// Two MMA-issuing warps: a thread waits ~55-80 cycles for each tcgen05.mma it issues, whatever
// the MMA's N up to 64 (~100 at N = 128), so with ~20-30 tokens per expert the issue rate of one
// thread bounds the MMAs; two threads taking alternate K chunks into separate accumulators
// issue twice as many.  A chunk too wide for two accumulators is split by its tokens instead
// (the same MMA count per thread, each of half the N).
constexpr int kProdWarp = kDecWarps, kIssueWarp = kDecWarps + 1, kProdBWarp = kDecWarps + 2,
              kIssue2Warp = kDecWarps + 3;
constexpr int kIssuers = 2;
constexpr int kMmaThreads = kDecThreads + 128;
// A chunk of at most kSplitMax tokens (and >= 2 K chunks) is split by K between the two
// issuers: the second's accumulator takes the upper half of each 128-column accumulator.
constexpr int kSplitTokens = kGroupTokens / 2;
constexpr int kSplitMax = 64;
static_assert(kSplitMax <= kSplitTokens, "a split chunk fits half an accumulator");
__device__ __forceinline__ bool split_issue(int npad, int KC) { return npad <= kSplitMax && KC >= 2; }
constexpr int kBRing = 4;             // activation tile stages
constexpr int kARing = 8;             // weight tile stages (in tensor memory)
constexpr int kSegRing = 4;           // code segment stages
constexpr uint32_t kCopies = 8;       // codebook copies: lane j of a quarter-warp reads copy j
constexpr uint32_t kCbBytes = kStages * kCodes * kCopies * 16;  // 96 KiB of fp16 rows
constexpr uint32_t kBBytes = kGroupTokens * kBK * 2;           // 16 KiB
constexpr uint32_t kGroupBytes = kStages * 512;                // one row group of a segment
constexpr uint32_t kGroupStride = kGroupBytes + 16;            // padded in shared memory
constexpr uint32_t kSegBytes = 8 * kGroupStride;               // 8 row groups x 3 stages x 32 vectors
constexpr uint32_t kOffCb = 0;
constexpr uint32_t kOffB = kOffCb + kCbBytes;
constexpr uint32_t kOffSeg = kOffB + kBRing * kBBytes;
constexpr uint32_t kOffSlot = kOffSeg + kSegRing * kSegBytes;
// two slot lists: the down kernel takes an item's epilogue under the next item's decode
constexpr uint32_t kOffBar = (kOffSlot + 2 * kGroupTokens * 4 + 7) & ~7u;
// barrier indices (two accumulators' full / empty pairs: gate/up uses the first only)
enum { kSegFull = 0, kSegEmpty = kSegRing, kBFull = 2 * kSegRing, kBEmpty = kBFull + kBRing, kAFull = kBEmpty + kBRing,
       kAEmpty = kAFull + kARing, kAccFull = kAEmpty + kARing, kAccEmpty = kAccFull + 2, kNumBars = kAccEmpty + 2 };
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kMmaSmem = kOffMisc + 16;
// tensor memory: [0, 256) the gate and up accumulators (128 columns each; down: two
// accumulators used by alternate items), [256, 512) the weight tiles (kARing x 32 columns:
// 128 rows x 64 fp16 weights each)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemA = 2 * kGroupTokens;
static_assert(kMmaSmem <= 227 * 1024, "shared memory of the tensor-core kernel");
static_assert(kTmemA + kARing * (kBK / 2) <= kTmemCols, "tensor memory of the tensor-core kernel");

struct MmaArgs {
    const uint8_t *records;
    const int32_t *slot_map;
    size_t stride;
    size_t sec[3];
    const float *codebooks;
    MatGeom geom; // the matrix of this kernel (gate/up: f x d, down: d x f)
    int d, f, k, nparts;
    const int32_t *sorted;
    const int4 *chunks;
    const int32_t *counts;
    const uint8_t *bsrc; // tiled fp16 activations the MMAs read (xg or ag)
    uint8_t *ag;         // gate/up output tiles (down input)
    float *part_dn;      // [S][nparts][d]
    unsigned long long *stats;
    uint32_t *err;
};

__device__ __forceinline__ uint32_t half2_bits(float a, float b) {
    const __half2 p = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&p);
}
__device__ __forceinline__ uint32_t hadd2_bits(uint32_t a, uint32_t b) {
    const __half2 r = __hadd2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Explicit shared-memory loads at 32-bit shared-window addresses (never generic accesses).
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void dec_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kDecThreads) : "memory"); }

// Wait for the phase of the given parity.  Gives up after a second (then raises the
// CTA's abort flag) or at once when the flag is already up; with check_abort false only
// the second bounds it (used to drain copies and MMAs in flight before exit).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           bool check_abort = true) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (check_abort && *abort_flag) return false;
            if (global_ns() - t0 > 1000000000ull) {
                *abort_flag = 1;
                return false;
            }
            __nanosleep(64);
        }
    }
}

// The same for a whole warp: every lane waits, lane 0's verdict counts for all.
__device__ __forceinline__ bool wait_phase_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                bool check_abort = true) {
    const bool ok = wait_phase(bar, parity, abort_flag, check_abort);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// The items of this CTA: a contiguous range of the (chunk, 128-row block) items, so that
// consecutive items mostly share their expert and its codebooks stay in shared memory.
__device__ __forceinline__ void cta_items(int n_items, int &i0, int &i1) {
    const int per = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;
    i0 = min(n_items, (int)blockIdx.x * per);
    i1 = min(n_items, i0 + per);
}

// Matrix of pass `pass` of the CTA's it-th item: down has one pass; gate/up alternate their
// order from item to item, so the last pass's codebooks serve the next item's first pass.
template <bool kDown>
__device__ __forceinline__ int pass_mat(int it, int pass) {
    if constexpr (kDown) return 2;
    return (pass ^ (it & 1));
}

// One item = (chunk of <= 128 tokens of one expert, 128-row block of the output).
// Weights are decoded from their codes into tensor memory (the MMA's A operand); the
// activation tiles come from shared memory (B operand).
template <bool kDown>
__global__ void __launch_bounds__(kMmaThreads, 1) mma_kernel(const MmaArgs A) {
    extern __shared__ __align__(1024) unsigned char gsm[];
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(gsm);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int *s_slot = reinterpret_cast<int *>(gsm + kOffSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gsm + kOffMisc + 4);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
    if (tid == 0) {
        for (int i = 0; i < kSegRing; ++i) {
            tc::mbar_init(bar(kSegFull + i), 1);
            tc::mbar_init(bar(kSegEmpty + i), kDecWarps);
        }
        // a stage is free, and an accumulator full, once both issuers have committed it (a
        // commit covers that issuer's own MMAs issued so far, or none)
        for (int i = 0; i < kBRing; ++i) {
            tc::mbar_init(bar(kBFull + i), 1);
            tc::mbar_init(bar(kBEmpty + i), kIssuers);
        }
        for (int i = 0; i < kARing; ++i) {
            tc::mbar_init(bar(kAFull + i), kDecWarps);
            tc::mbar_init(bar(kAEmpty + i), kIssuers);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(kAccFull + i), kIssuers);
            tc::mbar_init(bar(kAccEmpty + i), kDecWarps);
        }
        tc::mbar_init_fence();
        *abort_flag = 0;
    }
    if (warp == 0) tc::tmem_alloc(sbase + kOffMisc, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gsm + kOffMisc);

    const MatGeom G = A.geom;
    const int nmb = (G.n_out + kBM - 1) / kBM;
    const int KC = (G.n_in + kBK - 1) / kBK;
    const int n_items = A.counts[0] * nmb;
    int i0, i1;
    cta_items(n_items, i0, i1);
    constexpr int kPasses = kDown ? 1 : 2;

    if (warp == kProdWarp) {
        // ---------------- code producer: the codes of each 32-vector segment of the row
        // block, one bulk copy per row group into padded slots (the whole warp walks the loop;
        // lane 0 issues).  At the start of each (item, pass) the codes of the next one are
        // asked of L2, so the segment copies find them there.
        uint32_t gs = 0;
        auto l2_ahead = [&](int item, int pass) {
            if (item >= i1) return;
            const int4 c = A.chunks[item / nmb];
            const uint8_t *r = expert_record(A.records, A.stride, A.slot_map, c.x);
            if (!r) return;
            const int mb = item % nmb;
            const uint32_t bytes = (uint32_t)min(8, G.groups - 8 * mb) * kGroupBytes;
            const uint8_t *sec = r + A.sec[pass_mat<kDown>(item - i0, pass)];
            for (int sg = lane; sg < G.nseg; sg += 32) {
                const uint8_t *src = sec + ((size_t)sg * G.groups + 8 * mb) * kGroupBytes;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
            }
        };
        l2_ahead(i0, 0);
        for (int item = i0; item < i1; ++item) {
            const int4 ch = A.chunks[item / nmb];
            const int mb = item % nmb;
            const uint8_t *rec = expert_record(A.records, A.stride, A.slot_map, ch.x);
            if (!rec) {
                // not resident (a bank fetch did not place it): no copies, the row block
                // decodes whatever the buffers hold, and the error is latched
                if (lane == 0) atomicOr(A.err, kErrNotResident);
                rec = A.records;
            }
            const int n_groups = min(8, G.groups - 8 * mb);
            for (int pass = 0; pass < kPasses; ++pass) {
                if (pass + 1 < kPasses) l2_ahead(item, pass + 1);
                else l2_ahead(item + 1, 0);
                const uint8_t *sec = rec + A.sec[pass_mat<kDown>(item - i0, pass)];
                for (int kc0 = 0; kc0 < KC; kc0 += kKcSeg, ++gs) {
                    const int sb = gs % kSegRing;
                    const bool ok = gs < kSegRing ||
                                    wait_phase_warp(bar(kSegEmpty + sb), ((gs - kSegRing) / kSegRing) & 1, abort_flag);
                    if (ok && lane == 0 && !*abort_flag) {
                        const uint8_t *src = sec + ((size_t)(kc0 / kKcSeg) * G.groups + 8 * mb) * kGroupBytes;
                        tc::mbar_arrive_expect_tx(bar(kSegFull + sb), (uint32_t)n_groups * kGroupBytes);
                        for (int g = 0; g < n_groups; ++g)
                            tc::bulk_g2s(sbase + kOffSeg + sb * kSegBytes + g * kGroupStride, src + g * kGroupBytes,
                                         kGroupBytes, bar(kSegFull + sb));
                    }
                    __syncwarp();
                }
            }
        }
        // drain: the last copies into each buffer have landed before the CTA exits
        for (uint32_t i = 0; i < (uint32_t)kSegRing && i < gs; ++i) {
            const uint32_t g = gs - 1 - i;
            wait_phase_warp(bar(kSegFull + g % kSegRing), (g / kSegRing) & 1, abort_flag, false);
        }
    } else if (warp == kProdBWarp) {
        // ---------------- activation producer: the tile of each 64-wide K chunk
        uint32_t q = 0;
        for (int item = i0; item < i1; ++item) {
            const int4 ch = A.chunks[item / nmb];
            const uint32_t bbytes = (uint32_t)pad16(ch.z) * 128;
            const uint8_t *bsrc = A.bsrc + (size_t)ch.w * KC * 128;
            for (int pass = 0; pass < kPasses; ++pass) {
                for (int kc = 0; kc < KC; ++kc, ++q) {
                    const int rs = q % kBRing;
                    const bool ok = q < kBRing ||
                                    wait_phase_warp(bar(kBEmpty + rs), ((q - kBRing) / kBRing) & 1, abort_flag);
                    if (ok && lane == 0 && !*abort_flag) {
                        tc::mbar_arrive_expect_tx(bar(kBFull + rs), bbytes);
                        tc::bulk_g2s(sbase + kOffB + rs * kBBytes, bsrc + (size_t)kc * bbytes, bbytes, bar(kBFull + rs));
                    }
                    __syncwarp();
                }
            }
        }
        for (uint32_t i = 0; i < (uint32_t)kBRing && i < q; ++i) {
            const uint32_t g = q - 1 - i;
            wait_phase_warp(bar(kBFull + g % kBRing), (g / kBRing) & 1, abort_flag, false);
        }
    } else if (warp == kIssueWarp || warp == kIssue2Warp) {
        // ---------------- MMA issue (each issuing warp walks the loop; its lane 0 issues).  A
        // K-split item: the first issuer takes the even chunks of the CTA's chunk sequence, the
        // second the odd ones (every pass of >= 2 chunks gives each at least one), each into its
        // own accumulator.  Otherwise both take every chunk, the first for the accumulator
        // columns (tokens) [0, n0), the second for [n0, npad): B rows from n0 on, n0 a multiple
        // of 16 (the MMA's N for M = 128); a chunk of 16 tokens is the first issuer's alone.
        // Both wait for every stage and commit every stage and item, so neither runs more than a
        // ring ahead of the other or of the producers, and no parity wait is ever two phases off.
        const uint32_t mine = warp == kIssue2Warp ? 1u : 0u;
        uint32_t q = 0, it = 0;
        for (int item = i0; item < i1; ++item, ++it) {
            const int4 ch = A.chunks[item / nmb];
            const int npad = pad16(ch.z);
            const bool split = split_issue(npad, KC);
            const int n0 = npad >= 32 ? ((npad / 2 + 15) & ~15) : npad;
            const int c0 = split || mine == 0u ? 0 : n0;                 // first token column
            const int nb = split ? npad : (mine == 0u ? n0 : npad - n0); // 0 or a multiple of 16
            const uint32_t idesc = tc::idesc_f16_f32(kBM, nb > 0 ? nb : 16);
            // down: item it accumulates into buffer it & 1, free once item it - 2's epilogue is done
            const int ba = kDown ? (int)(it & 1) : 0;
            if (kDown ? it >= 2 : it >= 1)
                wait_phase_warp(bar(kAccEmpty + ba), kDown ? ((it - 2) >> 1) & 1 : (it - 1) & 1, abort_flag);
            tc::fence_after_sync();
            for (int pass = 0; pass < kPasses; ++pass) {
                const uint32_t acc = tmem + (uint32_t)(kDown ? ba : pass_mat<kDown>(it, pass)) * kGroupTokens +
                                     (split ? mine * (uint32_t)kSplitTokens : (uint32_t)c0);
                bool fresh = true; // this issuer's first chunk of the pass starts its accumulator
                for (int kc = 0; kc < KC; ++kc, ++q) {
                    const bool take = split ? (q & 1u) == mine : nb > 0;
                    const int ab = q % kARing, rs = q % kBRing;
                    wait_phase_warp(bar(kAFull + ab), (q / kARing) & 1, abort_flag);
                    wait_phase_warp(bar(kBFull + rs), (q / kBRing) & 1, abort_flag);
                    tc::fence_after_sync();
                    if (lane == 0) {
                        if (take) {
                            const uint32_t a_tm = tmem + kTmemA + (uint32_t)ab * (kBK / 2);
                            // B rows of 8 tokens are 1024 bytes apart (the descriptor's SBO)
                            const uint32_t b_addr = sbase + kOffB + rs * kBBytes + (uint32_t)(c0 / 8) * 1024;
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk)
                                tc::mma_f16_ta(acc, a_tm + kk * 8, tc::smem_desc(b_addr + kk * 256, 128, 1024),
                                               idesc, !fresh || kk != 0);
                        }
                        tc::mma_commit(bar(kAEmpty + ab));
                        tc::mma_commit(bar(kBEmpty + rs));
                    }
                    if (take) fresh = false;
                    __syncwarp();
                }
            }
            if (lane == 0) {
                tc::mma_commit(bar(kAccFull + ba));
                if (A.stats && mine == 0u) {
                    const int mb = item % nmb;
                    const int rows = min(G.n_out - mb * kBM, kBM);
                    atomicAdd(A.stats + kStatDemandCode, (unsigned long long)kPasses * rows * G.nv * kStages);
                    if (mb == 0)
                        atomicAdd(A.stats + kStatCodebook,
                                  (unsigned long long)kPasses * kStages * kCodes * kVec * sizeof(float));
                }
            }
            __syncwarp();
        }
        // drain: every MMA issued (by either issuer) has completed before TMEM is released
        if (it >= 1) {
            const uint32_t last = it - 1;
            wait_phase_warp(bar(kAccFull + (kDown ? (int)(last & 1) : 0)), kDown ? (last >> 1) & 1 : last & 1,
                            abort_flag, false);
        }
    } else {
        // ---------------- decode warps (and the epilogue).  Warp w writes the weight rows of
        // TMEM lane quarter w % 4 (rows 32 (w % 4) + lane of the block) for the K slice w / 4
        // of each 64-wide chunk: vectors 2 (w / 4) and 2 (w / 4) + 1 of the chunk's 8.
        const int lq = warp & 3, wg = warp >> 2;
        const int rl = lq * 32 + lane;                  // row of the 128-row block
        const int rr = rl & 15, gl = rl >> 4;           // row in its group, group in the block
        // shared-window address of this lane's codebook copy (stage 0, code 0)
        const uint32_t cb_lane = sbase + kOffCb + (uint32_t)(lane & 7) * 16;
        const uint32_t a_lane = (uint32_t)(lq * 32) << 16;
        int loaded = -1; // (expert * 3 + matrix) whose codebooks are in shared memory
        // An item's epilogue: warp w reads TMEM lanes 32 (w % 4) .. +32 (its output rows) and the
        // column blocks of 16 starting at 16 (w / 4), every 64.  Down: item j's accumulator is
        // buffer j & 1 and its slot list the list j & 1; it runs under the next item's decode.
        struct Ep {
            uint32_t j;
            int row, nt, npad;
            bool row_ok;
            int4 ch;
        };
        auto epilogue = [&](const Ep &E) {
            const int ba = kDown ? (int)(E.j & 1) : 0;
            wait_phase(bar(kAccFull + ba), kDown ? (E.j >> 1) & 1 : E.j & 1, abort_flag);
            tc::fence_after_sync();
            const int *slots = s_slot + (kDown ? ba * kGroupTokens : 0);
            const uint32_t lane_addr = tmem + a_lane + (uint32_t)ba * kGroupTokens;
            const int kcf = (A.f + kBK - 1) / kBK;
            uint8_t *ag = A.ag + (size_t)E.ch.w * kcf * 128;
            const int row = E.row, nt = E.nt, npad = E.npad;
            const bool split = split_issue(npad, KC);
            for (int c0 = wg * 16; c0 < npad; c0 += 64) {
                float z[16];
                tc::tmem_ld16(lane_addr + c0, z);
                if (split) {
                    float z2[16];
                    tc::tmem_ld16(lane_addr + kSplitTokens + c0, z2);
#pragma unroll
                    for (int n = 0; n < 16; ++n) z[n] += z2[n];
                }
                if constexpr (!kDown) {
                    float u[16];
                    tc::tmem_ld16(lane_addr + kGroupTokens + c0, u);
                    if (split) {
                        float u2[16];
                        tc::tmem_ld16(lane_addr + kGroupTokens + kSplitTokens + c0, u2);
#pragma unroll
                        for (int n = 0; n < 16; ++n) u[n] += u2[n];
                    }
                    if (E.row_ok) {
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            if (c0 + n < nt) {
                                const float a = z[n] / (1.0f + expf(-z[n])) * u[n];
                                const __half ha = __float2half_rn(a);
                                *reinterpret_cast<__half *>(ag + tile_off(row >> 6, npad, c0 + n, row) +
                                                            (row & 7) * 2) = ha;
                            }
                    }
                } else {
                    if (E.row_ok) {
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            if (c0 + n < nt) A.part_dn[(size_t)slots[c0 + n] * A.nparts * A.d + row] = z[n];
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(kAccEmpty + ba));
        };
        Ep pend_ep;
        bool have_ep = false;           // down: an epilogue waits for the next item's first chunks
        const int defer_at = min(kARing, KC); // chunks of an item decoded before it runs
        uint32_t q = 0, gs = 0, it = 0;
        for (int item = i0; item < i1; ++item, ++it) {
            const int4 ch = A.chunks[item / nmb];
            const int e = ch.x, nt = ch.z, npad = pad16(nt);
            const int mb = item % nmb;
            const int row = mb * kBM + rl;
            const bool row_ok = row < G.n_out;
            int *slots_it = s_slot + (kDown ? (int)(it & 1) * kGroupTokens : 0);
            int kc_item = 0; // chunks of this item decoded (down's deferred epilogue)
            for (int pass = 0; pass < kPasses; ++pass) {
                const int mat = pass_mat<kDown>(it, pass);
                const int key = e * 3 + mat;
                // the same for every decode thread: the down epilogue's slot list changes with
                // the item, the codebooks with the (expert, matrix)
                const bool new_slots = kDown && pass == 0, reload = key != loaded;
                if (new_slots || reload) {
                    dec_barrier(); // every decode warp is past the previous pass (and epilogue)
                    if (new_slots && tid < kGroupTokens) slots_it[tid] = tid < nt ? A.sorted[ch.y + tid] : 0;
                    if (reload) {
                        // codebook rows as fp16, 8 copies each; a thread writes its row's copies
                        // starting at its own, so a quarter-warp's stores hit 8 bank quads
                        const float *cb = A.codebooks + (size_t)key * (kStages * kCodes * kVec);
                        uint4 *dst = reinterpret_cast<uint4 *>(gsm + kOffCb);
                        for (int r = tid; r < kStages * kCodes; r += kDecThreads) {
                            const float4 lo = __ldg(reinterpret_cast<const float4 *>(cb) + 2 * r);
                            const float4 hi = __ldg(reinterpret_cast<const float4 *>(cb) + 2 * r + 1);
                            const uint4 hv = make_uint4(half2_bits(lo.x, lo.y), half2_bits(lo.z, lo.w),
                                                        half2_bits(hi.x, hi.y), half2_bits(hi.z, hi.w));
#pragma unroll
                            for (uint32_t c = 0; c < kCopies; ++c) dst[r * kCopies + ((c + r) & (kCopies - 1))] = hv;
                        }
                        loaded = key;
                    }
                    dec_barrier(); // codebook rows and slots in place
                }
                // a stage's tensor-memory stores are waited for one chunk later, so the decode of
                // the next chunk runs under them; `pend` is the stage still to be handed over
                int pend = -1;
                for (int kc0 = 0; kc0 < KC; kc0 += kKcSeg, ++gs) {
                    const int sb = gs % kSegRing;
                    wait_phase(bar(kSegFull + sb), (gs / kSegRing) & 1, abort_flag);
                    const uint32_t seg = sbase + kOffSeg + (uint32_t)sb * kSegBytes + (uint32_t)gl * kGroupStride;
                    for (int kc = kc0; kc < min(KC, kc0 + kKcSeg); ++kc, ++q) {
                        const int ab = q % kARing;
                        if (q >= kARing) {
                            wait_phase(bar(kAEmpty + ab), ((q - kARing) / kARing) & 1, abort_flag);
                            tc::fence_after_sync(); // the MMAs that read this stage are complete
                        }
                        // both vectors' codes first, then their codebook rows (the loads are
                        // volatile: issued in this order, all in flight before their uses)
                        uint32_t c[2][3];
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            const int jj = 8 * (kc - kc0) + 2 * wg + v; // vector within the segment
                            const uint32_t cp = seg + (uint32_t)(jj * 16 + ((rr ^ jj) & 15));
                            c[v][0] = lds_u8(cp);
                            c[v][1] = lds_u8(cp + 512);
                            c[v][2] = lds_u8(cp + 1024);
                        }
                        uint4 cv[2][3];
#pragma unroll
                        for (int v = 0; v < 2; ++v)
#pragma unroll
                            for (int st = 0; st < kStages; ++st)
                                cv[v][st] = lds_v4(cb_lane + ((uint32_t)st * kCodes + c[v][st]) * (kCopies * 16));
                        uint32_t w[8];
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            const int j = kc * 8 + 2 * wg + v; // vector within the row
                            const bool ok = row_ok && j < G.nv;
                            const uint4 &v0 = cv[v][0], &v1 = cv[v][1], &v2 = cv[v][2];
                            w[4 * v + 0] = ok ? hadd2_bits(hadd2_bits(v0.x, v1.x), v2.x) : 0u;
                            w[4 * v + 1] = ok ? hadd2_bits(hadd2_bits(v0.y, v1.y), v2.y) : 0u;
                            w[4 * v + 2] = ok ? hadd2_bits(hadd2_bits(v0.z, v1.z), v2.z) : 0u;
                            w[4 * v + 3] = ok ? hadd2_bits(hadd2_bits(v0.w, v1.w), v2.w) : 0u;
                        }
                        tc::tmem_st8(tmem + a_lane + kTmemA + (uint32_t)ab * (kBK / 2) + (uint32_t)wg * 8, w);
                        if (pend >= 0) {
                            tc::tmem_wait_st(); // both stages' stores are complete
                            tc::fence_before_sync();
                            __syncwarp();
                            if (lane == 0) {
                                tc::mbar_arrive(bar(kAFull + pend));
                                tc::mbar_arrive(bar(kAFull + ab));
                            }
                            pend = -1;
                        } else {
                            pend = ab;
                        }
                        if (kDown && have_ep && ++kc_item == defer_at) {
                            // the MMAs have defer_at chunks of this item queued: the previous
                            // item's epilogue now (its stage handed over first)
                            if (pend >= 0) {
                                tc::tmem_wait_st();
                                tc::fence_before_sync();
                                __syncwarp();
                                if (lane == 0) tc::mbar_arrive(bar(kAFull + pend));
                                pend = -1;
                            }
                            epilogue(pend_ep);
                            have_ep = false;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(bar(kSegEmpty + sb)); // its codes are read
                }
                if (pend >= 0) {
                    tc::tmem_wait_st();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(bar(kAFull + pend));
                }
            }
            const Ep cur{it, row, nt, npad, row_ok, ch};
            if constexpr (kDown) {
                pend_ep = cur;
                have_ep = true;
            } else {
                epilogue(cur);
            }
        }
        if (have_ep) epilogue(pend_ep);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort_flag) atomicOr(A.err, kErrTimeout);
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kDown>
cudaError_t launch_mma(const MmaArgs &A, int num_sms, cudaStream_t s) {
    static SmemAttr attr;
    cudaError_t e = ensure_smem(attr, (const void *)mma_kernel<kDown>, (int)kMmaSmem);
    if (e != cudaSuccess) return e;
    mma_kernel<kDown><<<num_sms, kMmaThreads, kMmaSmem, s>>>(A);
    return cudaGetLastError();
}

} // namespace

size_t grouped_tile_rows(int max_slots, int max_chunks) {
    return (size_t)max_slots + 15 * (size_t)max_chunks;
}

cudaError_t launch_grouped_forward(const LayerView &L, const Workspace &W, const void *h, int T,
                                   const int32_t *idx, const float *gate, float *out, int mode,
                                   int min_tokens, bool reconstruct, int num_sms, cudaStream_t s,
                                   Timing *tm) {
    const Grouping &G = W.grp;
    const int S = T * L.k;
    if (tm) cudaEventRecord(tm->ev[0], s);
    group_kernel<<<1, kGroupThreads, 0, s>>>(idx, S, L.E, min_tokens < 1 ? 1 : min_tokens, G);
    if (L.act_bf16)
        gather_kernel<true><<<num_sms * 2, 256, 0, s>>>(h, G, L.d, L.f, L.k);
    else
        gather_kernel<false><<<num_sms * 2, 256, 0, s>>>(h, G, L.d, L.f, L.k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    MmaArgs A;
    A.records = L.records;
    A.slot_map = L.slot_map;
    A.stride = L.stride;
    for (int m = 0; m < 3; ++m) A.sec[m] = L.sec_off[m];
    A.codebooks = L.codebooks;
    A.d = L.d;
    A.f = L.f;
    A.k = L.k;
    A.nparts = down_parts(L);
    A.sorted = G.sorted;
    A.chunks = G.chunks;
    A.counts = G.counts;
    A.ag = G.ag;
    A.part_dn = W.part_dn;
    A.stats = W.stats;
    A.err = W.err;

    // gate/up: lookup slots, then the tensor-core chunks
    e = launch_lut_listed(L, W, h, T, idx, G.lut_slots, G.counts + 1, false, reconstruct, num_sms, s);
    if (e != cudaSuccess) return e;
    A.geom = L.gu;
    A.bsrc = G.xg;
    e = launch_mma<false>(A, num_sms, s);
    if (e != cudaSuccess) return e;
    if (tm) cudaEventRecord(tm->ev[1], s);
    // down
    e = launch_lut_listed(L, W, h, T, idx, G.lut_slots, G.counts + 1, true, reconstruct, num_sms, s);
    if (e != cudaSuccess) return e;
    A.geom = L.dn;
    A.bsrc = G.ag;
    e = launch_mma<true>(A, num_sms, s);
    if (e != cudaSuccess) return e;
    if (tm) cudaEventRecord(tm->ev[2], s);
    e = launch_combine(L, W, h, T, idx, gate, out, mode, G.one_part, A.nparts, s);
    if (e != cudaSuccess) return e;
    if (tm) {
        cudaEventRecord(tm->ev[3], s);
        tm->n = 4;
    }
    return cudaSuccess;
}

} // namespace wm
