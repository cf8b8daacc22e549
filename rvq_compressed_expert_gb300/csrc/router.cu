// Router GEMV/GEMM, top-k with gate normalisation, and the L2 prefetch of
// predicted experts.
//
// Routing: every token picks its experts from the router logits W_r h (+ b);
// the pages' model keeps 16 expert IDs per token and layer (page "Exécuter
// Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée et
// prédiction du routeur").  Order: logit descending, lowest index first on
// equal logits; gates: softmax over the k selected logits.
#include "route_dev.cuh"
#include "tc_dev.cuh"

#include <algorithm>

namespace wm {

using namespace route;

namespace {

// Small-T router: 2 experts per CTA of 256 threads.
constexpr int kRouterRows = 2;

template <bool kBf16>
__global__ void __launch_bounds__(256) router_small_kernel(const float *__restrict__ W,
                                                           const float *__restrict__ bias,
                                                           const void *__restrict__ h, int T,
                                                           int E, int d,
                                                           float *__restrict__ logits,
                                                           float *__restrict__ logits_lo) {
    __shared__ float red[kRouterRows][4][kRouterTok];
    router_block<kBf16>(W, bias, h, T, E, d, blockIdx.x * kRouterRows, logits, logits_lo, red);
}

// Larger T: 64 tokens x 64 experts per CTA, 256 threads with 4x4 outputs each,
// K staged through shared memory 32 at a time.
constexpr int kTileT = 64, kTileE = 64, kTileK = 32;

template <bool kBf16>
__global__ void __launch_bounds__(256) router_tiled_kernel(const float *__restrict__ W,
                                                           const float *__restrict__ bias,
                                                           const void *__restrict__ h, int T,
                                                           int E, int d,
                                                           float *__restrict__ logits,
                                                           float *__restrict__ logits_lo) {
    __shared__ float Hs[kTileK][kTileT + 4];
    __shared__ float Ws[kTileK][kTileE + 4];
    const int t0 = blockIdx.y * kTileT, e0 = blockIdx.x * kTileE;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4; // 16 x 16 threads
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
    for (int k0 = 0; k0 < d; k0 += kTileK) {
        // 64 rows x 32 k of each operand; 256 threads x 8 elements
        for (int i = threadIdx.x; i < kTileT * kTileK; i += 256) {
            const int r = i / kTileK, kk = i % kTileK;
            const int t = t0 + r, kg = k0 + kk;
            Hs[kk][r] = (t < T && kg < d) ? load_h1<kBf16>(h, (size_t)t * d + kg) : 0.f;
            const int e = e0 + r;
            Ws[kk][r] = (e < E && kg < d) ? W[(size_t)e * d + kg] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kTileK; ++kk) {
            float hv[4], wv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) hv[a] = Hs[kk][ty * 4 + a];
#pragma unroll
            for (int b = 0; b < 4; ++b) wv[b] = Ws[kk][tx * 4 + b];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(hv[a], wv[b], acc[a][b]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int t = t0 + ty * 4 + a;
        if (t >= T) continue;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int e = e0 + tx * 4 + b;
            if (e < E) {
                float hi = acc[a][b], lo = 0.f;
                if (bias) two_sum(acc[a][b], bias[e], hi, lo);
                logits[(size_t)t * E + e] = hi;
                if (logits_lo) logits_lo[(size_t)t * E + e] = lo;
            }
        }
    }
}

// Larger T, split along K: CTA (E tile, T tile, split) sums the products of its K range
// into part[split][t][e]; reduce_router_kernel adds the splits in order (then the bias,
// with its TwoSum remainder).  Tiles of 64 tokens x 64 experts, 256 threads with 4x4
// outputs each, K staged 32 at a time with 128-bit loads.
template <bool kBf16>
__global__ void __launch_bounds__(256) router_splitk_kernel(const float *__restrict__ W,
                                                            const void *__restrict__ h, int T, int E,
                                                            int d, int k_per_split,
                                                            float *__restrict__ part) {
    __shared__ float Hs[kTileK][kTileT + 4];
    __shared__ float Ws[kTileK][kTileE + 4];
    const int t0 = blockIdx.y * kTileT, e0 = blockIdx.x * kTileE;
    const int kb = blockIdx.z * k_per_split, ke = min(d, kb + k_per_split);
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
    // loader role: row r (of 64), 4-element group c4 (of 8), two rows per thread
    const int lr = threadIdx.x >> 3, lc = (threadIdx.x & 7) * 4;
    for (int k0 = kb; k0 < ke; k0 += kTileK) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = lr + 32 * half;
            const int kg = k0 + lc;
            const int t = t0 + r, e = e0 + r;
            // d % 8 == 0 and k ranges start at multiples of 32: a group of 4 is all in or out
            float4 hv = make_float4(0.f, 0.f, 0.f, 0.f), wv = hv;
            if (t < T && kg < ke) hv = load_h4<kBf16>(h, (size_t)t * d + kg);
            if (e < E && kg < ke) wv = *reinterpret_cast<const float4 *>(W + (size_t)e * d + kg);
            Hs[lc + 0][r] = hv.x;
            Hs[lc + 1][r] = hv.y;
            Hs[lc + 2][r] = hv.z;
            Hs[lc + 3][r] = hv.w;
            Ws[lc + 0][r] = wv.x;
            Ws[lc + 1][r] = wv.y;
            Ws[lc + 2][r] = wv.z;
            Ws[lc + 3][r] = wv.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kTileK; ++kk) {
            float hv[4], wv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) hv[a] = Hs[kk][ty * 4 + a];
#pragma unroll
            for (int b = 0; b < 4; ++b) wv[b] = Ws[kk][tx * 4 + b];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(hv[a], wv[b], acc[a][b]);
        }
        __syncthreads();
    }
    float *p = part + (size_t)blockIdx.z * T * E;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int t = t0 + ty * 4 + a;
        if (t >= T) continue;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int e = e0 + tx * 4 + b;
            if (e < E) p[(size_t)t * E + e] = acc[a][b];
        }
    }
}

__global__ void reduce_router_kernel(const float *__restrict__ part, int nsplit, const float *__restrict__ bias,
                                     int T, int E, float *__restrict__ logits, float *__restrict__ logits_lo) {
    const size_t n = (size_t)T * E;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        for (int sp = 0; sp < nsplit; ++sp) v += part[(size_t)sp * n + i];
        float hi = v, lo = 0.f;
        if (bias) two_sum(v, bias[i % E], hi, lo);
        logits[i] = hi;
        if (logits_lo) logits_lo[i] = lo;
    }
}

// Small-T router with the tokens staged in shared memory: 4 experts per CTA of 512
// threads, every lane's W_r loads in flight at once (same sums as the step kernel's
// router items).
// kRows expert rows per CTA (128 threads each).  With F.done set, the last CTA to finish its
// rows (a counter, zero at rest, put back by that CTA) also takes the top-k and gates of
// every token, in the kernel's shared memory: the routing in one launch.
template <bool kBf16, int kRows>
__global__ void __launch_bounds__(128 * kRows) router_staged_kernel(const float *__restrict__ W,
                                                                    const float *__restrict__ bias,
                                                                    const void *__restrict__ h, int T, int E,
                                                                    int d, float *__restrict__ logits,
                                                                    float *__restrict__ logits_lo,
                                                                    int hs_tokens, const RouteTopk F) {
    extern __shared__ __align__(16) float hs_dyn[];
    __shared__ float red[kRows][4][kRouterTok];
    __shared__ int last;
    router_block_staged<kBf16>(W, bias, h, T, E, d, blockIdx.x * kRows, logits, logits_lo, red, hs_dyn,
                               hs_tokens);
    if (!F.done) return;
    __threadfence(); // this CTA's logits before its count
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(F.done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence(); // every CTA's logits after their counts
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(hs_dyn);
    for (int t = 0; t < T; ++t)
        topk_block(logits, logits_lo, E, F.k, t, F.idx, F.gate, F.pred_idx, F.pred_count, F.pred_stride, F.stats,
                   F.router_bytes, keys, reinterpret_cast<int *>(keys + 512));
    if (threadIdx.x == 0) *F.done = 0u;
}

// Adds one to a counter with acquire-release semantics at GPU scope and returns the old value:
// the calling CTA's writes ordered before it by a barrier are published with it, and every
// CTA that counted before is visible after it.
__device__ __forceinline__ unsigned count_acq_rel(unsigned *c) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(c) : "memory");
    return old;
}

__device__ __forceinline__ unsigned long long route_gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// The top-k CTA of the polled one-token router: thread i waits (bounded, about a second) for
// expert i's selection key in slots[i] (0 = not yet written; one 64-bit store by the CTA that
// owns the row, read as one), clears the slot for the next call, and the CTA selects and
// gates (each warp sorts its 32 candidates, the lists are merged pairwise, as topk_block
// does).  While the row CTAs still work, a first pass runs the same selection on placeholder
// keys and stores nothing: only this CTA runs that code, which otherwise comes cold from
// memory (measured on GB300: the selection 0.6 us faster after the pass).  If a key never arrives, the timeout is latched, the token's experts are set
// to -1 (no expert: its slots contribute nothing) and no gates are formed.
__device__ __forceinline__ void route_poll_topk(int E, const RouteTopk F, uint32_t *err, unsigned long long *lk,
                                                int *li) {
    // warp 0 asks for the token's predicted experts now; they arrive during the wait
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int P = 0, pred_l = -1;
    if (warp == 0 && F.pred_count != nullptr) {
        P = F.pred_count[0];
        if (lane < F.pred_stride && lane < P) pred_l = F.pred_idx[lane];
    }
    const int i = threadIdx.x;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const bool real = pass == 1;
        Cand c;
        c.key = 0ull;
        c.id = 0x7fffffff;
        bool got = true;
        if (i < E) {
            unsigned long long v = 1ull + (unsigned long long)i; // placeholder key of the first pass
            if (real) {
                const unsigned long long t0 = route_gtimer();
                while ((v = ld_relaxed_u64(F.slots + i)) == 0ull) {
                    if (route_gtimer() - t0 > 1000000000ull) {
                        got = false;
                        break;
                    }
                }
                if (got) st_relaxed_u64(F.slots + i, 0ull);
            }
            if (got) {
                c.key = v;
                c.id = i;
            }
        }
        if (!__syncthreads_and(got ? 1 : 0)) {
            if (threadIdx.x == 0 && err) atomicOr(err, kErrTimeout);
            if (threadIdx.x < F.k) {
                F.idx[threadIdx.x] = -1;
                F.gate[threadIdx.x] = 0.f;
            }
            return;
        }
        warp_sort32(c);
        merge_warp_lists(c, lk, li);
        topk_emit(lk, li, F.k, 0, F.idx, F.gate, P, pred_l, F.pred_count, F.stats, F.router_bytes, real);
    }
}

// One token (decode): kRows expert rows per CTA of 128 threads (4 warps) per row.  Thread 0
// moves the rows of W_r and the token's h into shared memory with bulk copies (all of the
// rows' bytes in flight at once); the lanes then form router_block_staged's products in its
// order (per lane the float4s sub * 32 + lane + 128 u in turn, the warp's xor tree, the 4
// warps' sums in order), so the logits equal the staged kernel's bit for bit.  With F.done
// set, the last CTA to count itself also takes the top-k and gates; the count is one
// acquire-release atomic (no separate fences).  A copy that does not land within the
// bounded wait sets kErrTimeout in err; the CTA still counts itself, so the counter comes
// back to rest.  kPoll (a cooperative launch: every CTA resident at once): the row CTAs
// instead store each row's selection key into F.slots, and one more CTA (the last) waits for
// them and takes the top-k (route_poll_topk): no counter round trip, no re-read of the logits.
template <bool kBf16, int kRows, bool kPoll>
__global__ void __launch_bounds__(128 * kRows) router_t1_kernel(const float *__restrict__ W,
                                                                const float *__restrict__ bias,
                                                                const void *__restrict__ h, int E, int d,
                                                                float *__restrict__ logits,
                                                                float *__restrict__ logits_lo, const RouteTopk F,
                                                                uint32_t *err) {
    constexpr int kBig = 16;
    extern __shared__ __align__(16) unsigned char t1_smem[];
    __shared__ __align__(8) unsigned long long bar;
    __shared__ float red[kRows][4];
    __shared__ unsigned long long keys[128 * kRows];
    __shared__ int ids[128 * kRows];
    __shared__ int last;
    if constexpr (kPoll) {
        if (blockIdx.x == gridDim.x - 1) {
            route_poll_topk(E, F, err, keys, ids);
            return;
        }
    }
    // the CTAs past this layer's rows take the next layer's rows (F.ahead_w: the lookahead)
    const int grid1 = (E + kRows - 1) / kRows;
    const bool ahead = kPoll && (int)blockIdx.x >= grid1;
    if (ahead) {
        W = F.ahead_w;
        bias = F.ahead_b;
    }
    const int row0 = (ahead ? (int)blockIdx.x - grid1 : (int)blockIdx.x) * kRows;
    const int rows = min(kRows, (ahead ? F.ahead_E : E) - row0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rl = warp >> 2, sub = warp & 3;
    const uint32_t wbytes = (uint32_t)d * 4u, hbytes = (uint32_t)d * (kBf16 ? 2u : 4u);
    const unsigned char *hs = t1_smem + (size_t)kRows * wbytes;
    const uint32_t mb = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(mb, 1);
        tc::mbar_init_fence();
        tc::mbar_arrive_expect_tx(mb, (uint32_t)rows * wbytes + hbytes);
        const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(t1_smem);
        tc::bulk_g2s(s0 + (uint32_t)kRows * wbytes, h, hbytes, mb);
        for (int r = 0; r < rows; ++r) tc::bulk_g2s(s0 + (uint32_t)r * wbytes, W + (size_t)(row0 + r) * d, wbytes, mb);
    }
    __syncthreads(); // the barrier is initialised
    bool landed = tc::mbar_wait(mb, 0);
    if (!landed) {
        if (err) atomicOr(err, kErrTimeout);
        landed = tc::mbar_wait(mb, 0); // the copies in flight target this CTA's shared memory
    }
    landed = __syncthreads_and(landed ? 1 : 0) != 0; // one verdict for the whole CTA
    if (!landed) {
        // The copies never landed: the staged rows are not to be read.  No logits are
        // written; the CTA still counts itself so the counter returns to rest, and the last
        // CTA leaves the top-k alone (the timeout is latched; the copies may still be in
        // flight, so the context is to be treated as unusable).  Polled: the top-k CTA's wait
        // for this CTA's keys runs out instead.
        if (kPoll || !F.done) return;
        __syncthreads();
        if (threadIdx.x == 0 && count_acq_rel(F.done) == gridDim.x - 1) *F.done = 0u;
        return;
    }
    const float4 *ws = reinterpret_cast<const float4 *>(t1_smem + (size_t)rl * wbytes);
    const int d4 = d >> 2;
    const int per_lane = (d4 + 127) / 128;
    float acc = 0.f;
    if (rl < rows) {
        for (int m0 = 0; m0 < per_lane; m0 += kBig) {
#pragma unroll
            for (int u = 0; u < kBig; ++u) {
                const int i4 = sub * 32 + lane + 128 * (m0 + u);
                const int ic = min(i4, d4 - 1);
                const float4 w = ws[ic];
                float4 x;
                if constexpr (kBf16) {
                    const uint2 raw = reinterpret_cast<const uint2 *>(hs)[ic];
                    const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
                    const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
                    x = make_float4(fa.x, fa.y, fb.x, fb.y);
                } else {
                    x = reinterpret_cast<const float4 *>(hs)[ic];
                }
                float p = w.x * x.x;
                p = fmaf(w.y, x.y, p);
                p = fmaf(w.z, x.z, p);
                p = fmaf(w.w, x.w, p);
                acc = fmaf(i4 < d4 ? 1.f : 0.f, p, acc);
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) red[rl][sub] = acc;
    __syncthreads();
    if (threadIdx.x < rows) {
        const int r = row0 + (int)threadIdx.x;
        const float *q = red[threadIdx.x];
        const float v = ((q[0] + q[1]) + q[2]) + q[3];
        float hi = v, lo = 0.f;
        if (bias) two_sum(v, bias[r], hi, lo);
        if (ahead) {
            F.ahead_keys[r] = cand_key(hi, lo);
        } else {
            logits[r] = hi;
            if (logits_lo) logits_lo[r] = lo;
            if constexpr (kPoll) st_relaxed_u64(F.slots + r, cand_key(hi, lo));
        }
    }
    if (kPoll || !F.done) return;
    __syncthreads(); // this CTA's logits before its count
    if (threadIdx.x == 0) {
        last = count_acq_rel(F.done) == gridDim.x - 1;
        // some CTA's rows never arrived (the timeout it latched precedes its count): its
        // logits are missing, so the last CTA takes no top-k
        if (last && err && (atomicOr(err, 0u) & kErrTimeout)) {
            *F.done = 0u;
            last = 0;
        }
    }
    __syncthreads();
    if (!last) return;
    topk_block(logits, logits_lo, E, F.k, 0, F.idx, F.gate, F.pred_idx, F.pred_count, F.pred_stride, F.stats,
               F.router_bytes, keys, ids);
    if (threadIdx.x == 0) *F.done = 0u;
}

// Top-k of one token per CTA of 512 threads: per-warp sorted candidate lists merged in a
// tree (same selection and gates as the step kernel's top-k item).
__global__ void __launch_bounds__(512) topk_cta_kernel(const float *__restrict__ logits,
                                                       const float *__restrict__ logits_lo, int E,
                                                       int k, int32_t *__restrict__ idx,
                                                       float *__restrict__ gate,
                                                       const int32_t *__restrict__ pred_idx,
                                                       int32_t *__restrict__ pred_count,
                                                       int pred_stride,
                                                       unsigned long long *__restrict__ stats,
                                                       unsigned long long router_bytes) {
    extern __shared__ unsigned long long keys_dyn[];
    topk_block(logits, logits_lo, E, k, blockIdx.x, idx, gate, pred_idx, pred_count, pred_stride,
               stats, router_bytes, keys_dyn, reinterpret_cast<int *>(keys_dyn + 512));
}

// One warp per token.
__global__ void __launch_bounds__(32) topk_kernel(const float *__restrict__ logits,
                                                  const float *__restrict__ logits_lo, int E, int k,
                                                  int32_t *__restrict__ idx,
                                                  float *__restrict__ gate,
                                                  const int32_t *__restrict__ pred_idx,
                                                  int32_t *__restrict__ pred_count,
                                                  int pred_stride,
                                                  unsigned long long *__restrict__ stats,
                                                  unsigned long long router_bytes) {
    extern __shared__ float smem_topk[];
    topk_warp(logits, logits_lo, E, k, blockIdx.x, idx, gate, pred_idx, pred_count, pred_stride,
              stats, router_bytes, smem_topk);
}

// L2 prefetch of predicted experts: one CTA per (token, rank), the pieces of lookahead_piece.
__global__ void __launch_bounds__(128) prefetch_l2_kernel(const uint8_t *__restrict__ records, size_t stride,
                                                          size_t off_gate, size_t off_up, int nseg, int groups,
                                                          const float *__restrict__ codebooks, int E,
                                                          const int32_t *__restrict__ pred_idx,
                                                          int pred_stride, int P,
                                                          unsigned long long *stats) {
    const int t = blockIdx.x / P, p = blockIdx.x % P;
    const int e = pred_idx[(size_t)t * pred_stride + p];
    if (e < 0 || e >= E) return;
    for (int i = threadIdx.x; i < lookahead_pieces(nseg); i += blockDim.x)
        lookahead_piece(records, stride, off_gate, off_up, nseg, groups, codebooks, e, i);
    if (threadIdx.x == 0 && stats) {
        atomicAdd(stats + kStatPrefetchBytes, lookahead_bytes(nseg, groups));
        atomicAdd(stats + kStatPrefetchExperts, 1ull);
    }
}

// Weightless RMS normalisation of one token per CTA: out = in / sqrt(mean(in^2) + 1e-6),
// with the sum of squares reduced in a fixed order.
__global__ void __launch_bounds__(1024) rmsnorm_kernel(const float *__restrict__ in,
                                                       float *__restrict__ out, int d) {
    __shared__ float part[32];
    const float *x = in + (size_t)blockIdx.x * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (threadIdx.x == 0) part[0] = v;
    }
    __syncthreads();
    const float scale = 1.0f / sqrtf(part[0] / (float)d + 1e-6f);
    for (int i = threadIdx.x; i < d; i += blockDim.x) out[(size_t)blockIdx.x * d + i] = x[i] * scale;
}

__global__ void set_count_kernel(int32_t *count, int T, int P) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < T) count[t] = P;
}

} // namespace

constexpr size_t kRouterStageMax = 200 * 1024; // shared memory for staged hidden states

// Expert rows per CTA of the staged router (measured on GB300 at E = 384: four rows per
// CTA of 512 threads ran faster than two per CTA of 256).
constexpr int kStagedRows = 4;
// Expert rows per CTA of the one-token router, and its shared memory (the rows of W_r and h):
// up to d = 10,240 with fp32 hidden states.
#ifndef WM_T1_ROWS
#define WM_T1_ROWS 3
#endif
constexpr int kT1Rows = WM_T1_ROWS;
constexpr size_t kT1SmemMax = 160 * 1024;

static bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// Whether `ctas` CTAs of the one-token router can all be resident at once on the current
// device (one per SM: each holds over 100 KiB of shared memory) and the device takes
// cooperative launches: the polled form's top-k CTA waits for the others.
static bool t1_poll_fits(int ctas, int num_sms);

bool route_polled_fits(const LayerView &L, const void *h, int T, int ahead_E, int num_sms) {
    const size_t t1_smem = (size_t)L.d * (4 * kT1Rows + (L.act_bf16 ? 2 : 4));
    const int ctas = (L.E + kT1Rows - 1) / kT1Rows + (ahead_E + kT1Rows - 1) / kT1Rows + 1;
    return T == 1 && (size_t)L.d * 4 <= kRouterStageMax && t1_smem <= kT1SmemMax && aligned16(L.router_w) &&
           aligned16(h) && L.E <= 128 * kT1Rows && t1_poll_fits(ctas, num_sms);
}

static bool t1_poll_fits(int ctas, int num_sms) {
    static std::atomic<int> coop[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    int c = coop[dev].load(std::memory_order_acquire);
    if (c == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) v = 0;
        c = v ? 1 : 2;
        coop[dev].store(c, std::memory_order_release);
    }
    return c == 1 && ctas <= num_sms;
}

int router_splits(int T, int E, int d, int num_sms) {
    const int tiles = ((E + kTileE - 1) / kTileE) * ((T + kTileT - 1) / kTileT);
    int ns = (2 * num_sms + tiles - 1) / tiles;
    const int max_ns = (d + 255) / 256; // at least 256 of K per split
    if (ns > max_ns) ns = max_ns;
    if (ns > kRouterMaxSplits) ns = kRouterMaxSplits;
    return ns < 1 ? 1 : ns;
}

cudaError_t launch_router(const LayerView &L, const void *h, int T, float *logits,
                          float *logits_lo, cudaStream_t s, float *part, int num_sms, const RouteTopk *fuse,
                          bool *fused, uint32_t *err) {
    const size_t row_bytes = (size_t)L.d * 4;
    if (fused) *fused = false;
    if (T <= 16 && row_bytes <= kRouterStageMax) {
        const int hs_tokens = (int)std::min<size_t>({(size_t)kRouterTok, (size_t)T, kRouterStageMax / row_bytes});
        // the staged tokens' space, which the last CTA reuses for the top-k's candidate lists
        const size_t smem = std::max((size_t)hs_tokens * row_bytes, (size_t)kStagedRows * 128 / 32 * 32 * 12);
        // one token (decode): the top-k rides on the router launch; more tokens keep the
        // top-k kernel, which takes them in parallel
        if (fuse && fused && T == 1) *fused = true;
        else fuse = nullptr;
        static SmemAttr attr_s[2];
        cudaError_t ea = ensure_smem(attr_s[L.act_bf16 ? 1 : 0],
                                     L.act_bf16 ? (const void *)router_staged_kernel<true, kStagedRows>
                                                : (const void *)router_staged_kernel<false, kStagedRows>,
                                     (int)kRouterStageMax);
        if (ea != cudaSuccess) return ea;
        // the one-token kernel only for the demand route (fuse): its CTAs hold ~113 KiB of
        // shared memory and cannot run beside the expert kernels, which the lookahead's router
        // (another stream, no fuse) does on the staged kernel's 28 KiB (the same logits)
        const size_t t1_smem = (size_t)L.d * (4 * kT1Rows + (L.act_bf16 ? 2 : 4));
        if (T == 1 && fuse && fused && t1_smem <= kT1SmemMax && aligned16(L.router_w) && aligned16(h)) {
            const RouteTopk F = *fuse;
            const int grid1 = (L.E + kT1Rows - 1) / kT1Rows;
            const int grid2 = F.ahead_w ? (F.ahead_E + kT1Rows - 1) / kT1Rows : 0;
            if (F.slots && L.E <= 128 * kT1Rows && t1_poll_fits(grid1 + grid2 + 1, num_sms)) {
                // polled: the row CTAs and one top-k CTA, resident together
                static SmemAttr attr_p[2];
                const void *kfn = L.act_bf16 ? (const void *)router_t1_kernel<true, kT1Rows, true>
                                             : (const void *)router_t1_kernel<false, kT1Rows, true>;
                ea = ensure_smem(attr_p[L.act_bf16 ? 1 : 0], kfn, (int)kT1SmemMax);
                if (ea != cudaSuccess) return ea;
                cudaLaunchConfig_t lc = {};
                lc.gridDim = dim3(grid1 + grid2 + 1);
                lc.blockDim = dim3(128 * kT1Rows);
                lc.dynamicSmemBytes = t1_smem;
                lc.stream = s;
                cudaLaunchAttribute at[1];
                at[0].id = cudaLaunchAttributeCooperative;
                at[0].val.cooperative = 1;
                lc.attrs = at;
                lc.numAttrs = 1;
                if (L.act_bf16)
                    return cudaLaunchKernelEx(&lc, router_t1_kernel<true, kT1Rows, true>, L.router_w, L.router_b, h,
                                              L.E, L.d, logits, logits_lo, F, err);
                return cudaLaunchKernelEx(&lc, router_t1_kernel<false, kT1Rows, true>, L.router_w, L.router_b, h,
                                          L.E, L.d, logits, logits_lo, F, err);
            }
            static SmemAttr attr_t1[2];
            ea = ensure_smem(attr_t1[L.act_bf16 ? 1 : 0],
                             L.act_bf16 ? (const void *)router_t1_kernel<true, kT1Rows, false>
                                        : (const void *)router_t1_kernel<false, kT1Rows, false>,
                             (int)kT1SmemMax);
            if (ea != cudaSuccess) return ea;
            if (L.act_bf16)
                router_t1_kernel<true, kT1Rows, false><<<grid1, 128 * kT1Rows, t1_smem, s>>>(
                    L.router_w, L.router_b, h, L.E, L.d, logits, logits_lo, F, err);
            else
                router_t1_kernel<false, kT1Rows, false><<<grid1, 128 * kT1Rows, t1_smem, s>>>(
                    L.router_w, L.router_b, h, L.E, L.d, logits, logits_lo, F, err);
            return cudaGetLastError();
        }
        dim3 grid((L.E + kStagedRows - 1) / kStagedRows);
        if (L.act_bf16)
            router_staged_kernel<true, kStagedRows><<<grid, 128 * kStagedRows, smem, s>>>(
                L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo, hs_tokens, fuse ? *fuse : RouteTopk{});
        else
            router_staged_kernel<false, kStagedRows><<<grid, 128 * kStagedRows, smem, s>>>(
                L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo, hs_tokens, fuse ? *fuse : RouteTopk{});
    } else if (T <= 16) {
        dim3 grid((L.E + kRouterRows - 1) / kRouterRows);
        if (L.act_bf16)
            router_small_kernel<true><<<grid, 256, 0, s>>>(L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo);
        else
            router_small_kernel<false><<<grid, 256, 0, s>>>(L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo);
    } else if (part) {
        const int ns = router_splits(T, L.E, L.d, num_sms);
        const int kps = ((L.d + ns - 1) / ns + kTileK - 1) / kTileK * kTileK;
        const int nsu = (L.d + kps - 1) / kps;
        dim3 grid((L.E + kTileE - 1) / kTileE, (T + kTileT - 1) / kTileT, nsu);
        if (L.act_bf16)
            router_splitk_kernel<true><<<grid, 256, 0, s>>>(L.router_w, h, T, L.E, L.d, kps, part);
        else
            router_splitk_kernel<false><<<grid, 256, 0, s>>>(L.router_w, h, T, L.E, L.d, kps, part);
        const size_t n = (size_t)T * L.E;
        const int rg = (int)std::min<size_t>((n + 255) / 256, (size_t)num_sms * 8);
        reduce_router_kernel<<<rg, 256, 0, s>>>(part, nsu, L.router_b, T, L.E, logits, logits_lo);
    } else {
        dim3 grid((L.E + kTileE - 1) / kTileE, (T + kTileT - 1) / kTileT);
        if (L.act_bf16)
            router_tiled_kernel<true><<<grid, 256, 0, s>>>(L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo);
        else
            router_tiled_kernel<false><<<grid, 256, 0, s>>>(L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo);
    }
    return cudaGetLastError();
}

cudaError_t launch_topk(const float *logits, const float *logits_lo, int T, int E, int k,
                        int32_t *idx, float *gate, const int32_t *pred_idx, int32_t *pred_count,
                        int pred_stride, unsigned long long *stats,
                        unsigned long long router_bytes, cudaStream_t s) {
    // scratch of the warp top-k: 32 candidates (8-byte key, 4-byte index) per warp
    topk_cta_kernel<<<T, 512, 512 * 12, s>>>(logits, logits_lo, E, k, idx, gate, pred_idx, pred_count,
                                             pred_stride, stats, router_bytes);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float *in, float *out, int T, int d, cudaStream_t s) {
    rmsnorm_kernel<<<T, 1024, 0, s>>>(in, out, d);
    return cudaGetLastError();
}

cudaError_t launch_set_pred_count(int32_t *pred_count, int T, int P, cudaStream_t s) {
    set_count_kernel<<<(T + 255) / 256, 256, 0, s>>>(pred_count, T, P);
    return cudaGetLastError();
}

cudaError_t launch_prefetch_l2(const LayerView &L, const int32_t *pred_idx, int pred_stride,
                               int T, int P, int32_t *pred_count, unsigned long long *stats,
                               cudaStream_t s) {
    prefetch_l2_kernel<<<T * P, 128, 0, s>>>(L.records, L.stride, L.sec_off[0], L.sec_off[1], L.gu.nseg,
                                             L.gu.groups, L.codebooks, L.E, pred_idx, pred_stride, P, stats);
    set_count_kernel<<<(T + 255) / 256, 256, 0, s>>>(pred_count, T, P);
    return cudaGetLastError();
}

} // namespace wm
