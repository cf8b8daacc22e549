// Router GEMV/GEMM, top-k with gate normalisation, and the L2 prefetch of
// predicted experts.
//
// Routing: every token picks its experts from the router logits W_r h (+ b);
// the pages' model keeps 16 expert IDs per token and layer (page "Exécuter
// Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée et
// prédiction du routeur").  Order: logit descending, lowest index first on
// equal logits; gates: softmax over the k selected logits.
#include "common.cuh"

#include <float.h>

namespace wm {

namespace {

template <bool kBf16>
__device__ __forceinline__ float4 load_h4(const void *h, size_t elem) {
    if constexpr (kBf16) {
        const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(h) + elem;
        uint2 raw = *reinterpret_cast<const uint2 *>(p);
        __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
        float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        return make_float4(fa.x, fa.y, fb.x, fb.y);
    } else {
        return *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(h) + elem);
    }
}

template <bool kBf16>
__device__ __forceinline__ float load_h1(const void *h, size_t elem) {
    if constexpr (kBf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(h)[elem]);
    else return reinterpret_cast<const float *>(h)[elem];
}

// hi + lo == a + b exactly (Knuth's TwoSum); keeps the part of the dot product
// that adding a large bias would round away, so gate ratios stay accurate.
__device__ __forceinline__ void two_sum(float a, float b, float &hi, float &lo) {
    hi = __fadd_rn(a, b);
    const float bb = __fsub_rn(hi, a);
    lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(b, bb));
}

// Small-T router: 2 experts per CTA, 4 warps per expert row (each takes every
// 4th float4 of the row, 8 loads in flight per lane), up to 8 tokens per pass
// sharing each W_r load.
constexpr int kRouterRows = 2;
constexpr int kRouterTok = 8;
constexpr int kRouterBatch = 8;

template <bool kBf16>
__global__ void __launch_bounds__(256) router_small_kernel(const float *__restrict__ W,
                                                           const float *__restrict__ bias,
                                                           const void *__restrict__ h, int T,
                                                           int E, int d,
                                                           float *__restrict__ logits,
                                                           float *__restrict__ logits_lo) {
    __shared__ float red[kRouterRows][4][kRouterTok];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_local = warp >> 2, sub = warp & 3;
    const int row = blockIdx.x * kRouterRows + row_local;
    const int d4 = d >> 2;
    const int per_lane = (d4 + 127) / 128;
    for (int t0 = 0; t0 < T; t0 += kRouterTok) {
        const int nt = min(kRouterTok, T - t0);
        float acc[kRouterTok];
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) acc[t] = 0.f;
        if (row < E) {
            const float4 *w4 = reinterpret_cast<const float4 *>(W + (size_t)row * d);
            for (int m0 = 0; m0 < per_lane; m0 += kRouterBatch) {
                float4 w[kRouterBatch];
#pragma unroll
                for (int u = 0; u < kRouterBatch; ++u) {
                    const int i4 = sub * 32 + lane + 128 * (m0 + u);
                    w[u] = (i4 < d4) ? __ldg(w4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kRouterBatch; ++u) {
                    const int i4 = sub * 32 + lane + 128 * (m0 + u);
                    if (i4 >= d4) continue;
#pragma unroll
                    for (int t = 0; t < kRouterTok; ++t) {
                        if (t < nt) {
                            const float4 x = load_h4<kBf16>(h, (size_t)(t0 + t) * d + (size_t)i4 * 4);
                            acc[t] = fmaf(w[u].x, x.x, acc[t]);
                            acc[t] = fmaf(w[u].y, x.y, acc[t]);
                            acc[t] = fmaf(w[u].z, x.z, acc[t]);
                            acc[t] = fmaf(w[u].w, x.w, acc[t]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[row_local][sub][t] = v;
        }
        __syncthreads();
        if (threadIdx.x < kRouterRows * kRouterTok) {
            const int rl = threadIdx.x / kRouterTok, t = threadIdx.x % kRouterTok;
            const int r = blockIdx.x * kRouterRows + rl;
            if (r < E && t < nt) {
                float v = ((red[rl][0][t] + red[rl][1][t]) + red[rl][2][t]) + red[rl][3][t];
                float hi = v, lo = 0.f;
                if (bias) two_sum(v, bias[r], hi, lo);
                logits[(size_t)(t0 + t) * E + r] = hi;
                if (logits_lo) logits_lo[(size_t)(t0 + t) * E + r] = lo;
            }
        }
        __syncthreads();
    }
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

// Routing order: larger logit first (hi, then the exact remainder lo), lower
// index on ties.
__device__ __forceinline__ bool ranks_before(float ha, float la, int ia, float hb, float lb, int ib) {
    if (ha != hb) return ha > hb;
    if (la != lb) return la > lb;
    return ia < ib;
}

// One warp per token.  Logits staged in shared memory; k rounds of a warp
// arg-max that skips taken experts; softmax over the k selected logits with
// the differences taken as (hi_i - hi_0) + (lo_i - lo_0).
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
    float *lv = smem_topk;
    float *lw = lv + E;
    unsigned char *taken = reinterpret_cast<unsigned char *>(lw + E);
    const int t = blockIdx.x, lane = threadIdx.x;
#pragma unroll 8
    for (int e = lane; e < E; e += 32) {
        // canonical keys make the order total: -0 equals +0, and a NaN (outside the
        // contract) ranks as -inf, so every lane agrees on each round's winner
        float vh = logits[(size_t)t * E + e];
        float vl = logits_lo ? logits_lo[(size_t)t * E + e] : 0.f;
        if (vh != vh) vh = -INFINITY;
        if (vh == 0.f) vh = 0.f;
        if (vl != vl || vl == 0.f) vl = 0.f;
        lv[e] = vh;
        lw[e] = vl;
        taken[e] = 0;
    }
    __syncwarp();
    constexpr int kNone = 0x7fffffff;
    // each lane keeps the best untaken expert of its stripe e = lane (mod 32); a round
    // picks the best head across the warp, and only the owning lane rescans its stripe
    float hh = 0.f, hl = 0.f;
    int hidx = kNone;
    auto rescan = [&]() {
        hidx = kNone;
#pragma unroll 4
        for (int e = lane; e < E; e += 32) {
            if (taken[e]) continue;
            const float vh = lv[e], vl = lw[e];
            if (hidx == kNone || ranks_before(vh, vl, e, hh, hl, hidx)) {
                hh = vh;
                hl = vl;
                hidx = e;
            }
        }
    };
    rescan();
    int my_idx = -1;
    float my_hi = 0.f, my_lo = 0.f;
    for (int r = 0; r < k; ++r) {
        float bh = hh, bl = hl;
        int bi = hidx;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float oh = __shfl_xor_sync(0xffffffffu, bh, o);
            const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != kNone && (bi == kNone || ranks_before(oh, ol, oi, bh, bl, bi))) {
                bh = oh;
                bl = ol;
                bi = oi;
            }
        }
        if (lane == r) {
            my_idx = bi;
            my_hi = bh;
            my_lo = bl;
        }
        if (bi != kNone && lane == (bi & 31)) {
            taken[bi] = 1;
            rescan();
        }
    }
    // softmax over the selected logits; rank 0 holds the largest
    const float h0 = __shfl_sync(0xffffffffu, my_hi, 0);
    const float l0 = __shfl_sync(0xffffffffu, my_lo, 0);
    const float diff = (lane == 0) ? 0.f : __fsub_rn(my_hi, h0) + __fsub_rn(my_lo, l0);
    float ex = (lane < k) ? expf(diff) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
        idx[(size_t)t * k + lane] = my_idx;
        gate[(size_t)t * k + lane] = ex / sum;
    }
    if (pred_count != nullptr) {
        const int P = pred_count[t];
        bool hit = false;
        if (lane < k)
            for (int p = 0; p < P; ++p) hit |= (pred_idx[(size_t)t * pred_stride + p] == my_idx);
        const unsigned hits = __popc(__ballot_sync(0xffffffffu, hit));
        __syncwarp();
        if (lane == 0) {
            if (P > 0) atomicAdd(stats + kStatPredHits, (unsigned long long)hits);
            pred_count[t] = 0;
        }
    }
    if (lane == 0 && stats) {
        atomicAdd(stats + kStatRoutedSlots, (unsigned long long)k);
        if (t == 0) atomicAdd(stats + kStatRouter, router_bytes);
    }
}

// L2 prefetch of predicted experts' records: one CTA per (token, rank);
// each thread names 64 KiB pieces of the record's three sections.
__global__ void __launch_bounds__(128) prefetch_l2_kernel(const uint8_t *__restrict__ records,
                                                          size_t stride, size_t payload_off,
                                                          size_t payload_bytes, int E,
                                                          const int32_t *__restrict__ pred_idx,
                                                          int pred_stride, int P,
                                                          unsigned long long *stats) {
    const int t = blockIdx.x / P, p = blockIdx.x % P;
    const int e = pred_idx[(size_t)t * pred_stride + p];
    if (e < 0 || e >= E) return;
    const uint8_t *base = records + (size_t)e * stride + payload_off;
    constexpr size_t kPiece = 65536;
    for (size_t off = (size_t)threadIdx.x * kPiece; off < payload_bytes; off += 128 * kPiece) {
        const uint32_t n = (uint32_t)min(kPiece, payload_bytes - off);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + off), "r"(n)
                     : "memory");
    }
    if (threadIdx.x == 0 && stats) {
        atomicAdd(stats + kStatPrefetchBytes, (unsigned long long)payload_bytes);
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

cudaError_t launch_router(const LayerView &L, const void *h, int T, float *logits,
                          float *logits_lo, cudaStream_t s) {
    if (T <= 16) {
        dim3 grid((L.E + kRouterRows - 1) / kRouterRows);
        if (L.act_bf16)
            router_small_kernel<true><<<grid, 256, 0, s>>>(L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo);
        else
            router_small_kernel<false><<<grid, 256, 0, s>>>(L.router_w, L.router_b, h, T, L.E, L.d, logits, logits_lo);
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
    const size_t smem = (size_t)E * 2 * sizeof(float) + (size_t)E;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((size_t)kMaxExperts * 9));
        attr_set = true;
    }
    topk_kernel<<<T, 32, smem, s>>>(logits, logits_lo, E, k, idx, gate, pred_idx, pred_count,
                                    pred_stride, stats, router_bytes);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float *in, float *out, int T, int d, cudaStream_t s) {
    rmsnorm_kernel<<<T, 1024, 0, s>>>(in, out, d);
    return cudaGetLastError();
}

cudaError_t launch_prefetch_l2(const LayerView &L, const int32_t *pred_idx, int pred_stride,
                               int T, int P, int32_t *pred_count, unsigned long long *stats,
                               cudaStream_t s) {
    const size_t payload_off = L.sec_off[0];
    const size_t payload_bytes = L.sec_off[2] + L.dn.chunk_bytes() - L.sec_off[0];
    prefetch_l2_kernel<<<T * P, 128, 0, s>>>(L.records, L.stride, payload_off, payload_bytes, L.E,
                                             pred_idx, pred_stride, P, stats);
    set_count_kernel<<<(T + 255) / 256, 256, 0, s>>>(pred_count, T, P);
    return cudaGetLastError();
}

} // namespace wm
