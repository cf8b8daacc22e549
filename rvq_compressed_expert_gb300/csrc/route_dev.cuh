// Device-side routing pieces (router GEMV rows, per-token top-k and softmax), shared by
// the routing kernels (router.cu) and the fused decode-step kernel (fused.cu).
#pragma once

#include "common.cuh"

#include <float.h>

namespace wm {
namespace route {

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

// Routing order: larger logit first (hi, then the exact remainder lo), lower
// index on ties.
__device__ __forceinline__ bool ranks_before(float ha, float la, int ia, float hb, float lb, int ib) {
    if (ha != hb) return ha > hb;
    if (la != lb) return la > lb;
    return ia < ib;
}

// Router logits of rows [row_base, row_base + blockDim.x / 128) for T tokens: 4 warps per
// expert row (each takes every 4th float4 of the row, 8 loads in flight per lane), up to
// 8 tokens per pass sharing each W_r load; partial sums meet in `red` in a fixed order.
constexpr int kRouterTok = 8;
constexpr int kRouterBatch = 8;
constexpr int kRouterMaxRows = 4;

template <bool kBf16>
__device__ __forceinline__ void router_block(const float *__restrict__ W, const float *__restrict__ bias,
                                             const void *__restrict__ h, int T, int E, int d,
                                             int row_base, float *__restrict__ logits,
                                             float *__restrict__ logits_lo,
                                             float (*red)[4][kRouterTok]) {
    const int rows_per_block = blockDim.x >> 7;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_local = warp >> 2, sub = warp & 3;
    const int row = row_base + row_local;
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
                // every load of the batch is issued before any is used: indices past the row
                // are clamped to its last float4 and their products masked to zero
                float4 w[kRouterBatch];
                float m[kRouterBatch];
#pragma unroll
                for (int u = 0; u < kRouterBatch; ++u) {
                    const int i4 = sub * 32 + lane + 128 * (m0 + u);
                    m[u] = i4 < d4 ? 1.f : 0.f;
                    w[u] = __ldg(w4 + min(i4, d4 - 1));
                }
#pragma unroll
                for (int t = 0; t < kRouterTok; ++t) {
                    if (t < nt) {
                        float4 x[kRouterBatch];
#pragma unroll
                        for (int u = 0; u < kRouterBatch; ++u) {
                            const int i4 = min(sub * 32 + lane + 128 * (m0 + u), d4 - 1);
                            x[u] = load_h4<kBf16>(h, (size_t)(t0 + t) * d + (size_t)i4 * 4);
                        }
#pragma unroll
                        for (int u = 0; u < kRouterBatch; ++u) {
                            float p = w[u].x * x[u].x;
                            p = fmaf(w[u].y, x[u].y, p);
                            p = fmaf(w[u].z, x[u].z, p);
                            p = fmaf(w[u].w, x[u].w, p);
                            acc[t] = fmaf(m[u], p, acc[t]);
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
        if (threadIdx.x < rows_per_block * kRouterTok) {
            const int rl = threadIdx.x / kRouterTok, t = threadIdx.x % kRouterTok;
            const int r = row_base + rl;
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

// Top-k and softmax of token t by one warp; `area` is this warp's shared scratch of
// E * 9 bytes.  Logits are staged with canonical keys (-0 equals +0; a NaN, outside the
// contract, ranks as -inf) so the order is total and every lane agrees on each round's
// winner.  Each lane keeps the best untaken expert of its stripe e = lane (mod 32); a
// round picks the best head across the warp, and only the owning lane rescans.
__device__ __forceinline__ void topk_warp(const float *__restrict__ logits,
                                          const float *__restrict__ logits_lo, int E, int k, int t,
                                          int32_t *__restrict__ idx, float *__restrict__ gate,
                                          const int32_t *__restrict__ pred_idx,
                                          int32_t *__restrict__ pred_count, int pred_stride,
                                          unsigned long long *__restrict__ stats,
                                          unsigned long long router_bytes, float *area) {
    float *lv = area;
    float *lw = lv + E;
    unsigned char *taken = reinterpret_cast<unsigned char *>(lw + E);
    const int lane = threadIdx.x & 31;
    const float *lrow = logits + (size_t)t * E;
    const float *lorow = logits_lo ? logits_lo + (size_t)t * E : lrow;
    for (int e0 = 0; e0 < E; e0 += 32 * 8) {
        // 8 loads of each array in flight per lane (indices clamped, stores masked)
        float vh[8], vl[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = min(e0 + 32 * u + lane, E - 1);
            vh[u] = lrow[e];
            vl[u] = lorow[e];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = e0 + 32 * u + lane;
            if (e < E) {
                // canonical keys make the order total: -0 equals +0, and a NaN (outside
                // the contract) ranks as -inf, so every lane agrees on each round's winner
                float a = vh[u], b = logits_lo ? vl[u] : 0.f;
                if (a != a) a = -INFINITY;
                if (a == 0.f) a = 0.f;
                if (b != b || b == 0.f) b = 0.f;
                lv[e] = a;
                lw[e] = b;
                taken[e] = 0;
            }
        }
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

// Router logits of 4 expert rows per CTA of 512 threads, for T tokens, with the tokens'
// hidden states staged in shared memory `hs` (room for `hs_tokens` rows of d floats):
// each lane loads all of its float4s of W_r at once (16 per lane per pass), then takes
// h from shared memory.  Same partial sums, in the same order, as router_block.
template <bool kBf16>
__device__ __forceinline__ void router_block_staged(const float *__restrict__ W,
                                                    const float *__restrict__ bias,
                                                    const void *__restrict__ h, int T, int E, int d,
                                                    int row_base, float *__restrict__ logits,
                                                    float *__restrict__ logits_lo,
                                                    float (*red)[4][kRouterTok], float *hs,
                                                    int hs_tokens) {
    constexpr int kBig = 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_local = warp >> 2, sub = warp & 3;
    const int row = row_base + row_local;
    const int d4 = d >> 2;
    const int per_lane = (d4 + 127) / 128;
    const float4 *w4 = reinterpret_cast<const float4 *>(W + (size_t)min(row, E - 1) * d);
    for (int t0 = 0; t0 < T; t0 += kRouterTok) {
        const int nt = min(kRouterTok, T - t0);
        float acc[kRouterTok];
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) acc[t] = 0.f;
        for (int m0 = 0; m0 < per_lane; m0 += kBig) {
            float4 w[kBig];
            float m[kBig];
#pragma unroll
            for (int u = 0; u < kBig; ++u) {
                const int i4 = sub * 32 + lane + 128 * (m0 + u);
                m[u] = i4 < d4 ? 1.f : 0.f;
                w[u] = __ldg(w4 + min(i4, d4 - 1));
            }
            for (int tb = 0; tb < nt; tb += hs_tokens) {
                const int ntb = min(hs_tokens, nt - tb);
                __syncthreads(); // hs free
                for (int i = threadIdx.x; i < ntb * d4; i += blockDim.x) {
                    const int tt = i / d4, j = i % d4;
                    reinterpret_cast<float4 *>(hs)[i] = load_h4<kBf16>(h, (size_t)(t0 + tb + tt) * d + (size_t)j * 4);
                }
                __syncthreads();
#pragma unroll
                for (int t = 0; t < kRouterTok; ++t) {
                    if (t >= tb && t < tb + ntb) {
                        const float4 *x4 = reinterpret_cast<const float4 *>(hs) + (size_t)(t - tb) * d4;
#pragma unroll
                        for (int u = 0; u < kBig; ++u) {
                            const int i4 = min(sub * 32 + lane + 128 * (m0 + u), d4 - 1);
                            const float4 x = x4[i4];
                            float p = w[u].x * x.x;
                            p = fmaf(w[u].y, x.y, p);
                            p = fmaf(w[u].z, x.z, p);
                            p = fmaf(w[u].w, x.w, p);
                            acc[t] = fmaf(m[u], p, acc[t]);
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
        if (threadIdx.x < (int)(blockDim.x >> 7) * kRouterTok) {
            const int rl = threadIdx.x / kRouterTok, t = threadIdx.x % kRouterTok;
            const int r = row_base + rl;
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

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// Its inverse: the float whose key is k.
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// A routing candidate: 64-bit key (total-order image of the logit, then of its
// remainder) and the expert index; a comes before b in the selection order when its key
// is larger, or equal with a lower index.
struct Cand {
    unsigned long long key;
    int id;
};
__device__ __forceinline__ bool cand_before(const Cand &a, const Cand &b) {
    return a.key > b.key || (a.key == b.key && a.id < b.id);
}
__device__ __forceinline__ Cand shfl_cand(const Cand &c, int src) {
    Cand o;
    o.key = __shfl_sync(0xffffffffu, c.key, src);
    o.id = __shfl_sync(0xffffffffu, c.id, src);
    return o;
}
// One compare-exchange step of a bitonic network across the warp: lanes l and l ^ stride
// meet; the lower lane keeps the earlier candidate when `first_low`, else the later one.
__device__ __forceinline__ void bitonic_step(Cand &v, int stride, bool first_low) {
    const int lane = threadIdx.x & 31;
    const Cand o = shfl_cand(v, lane ^ stride);
    const bool low = (lane & stride) == 0;
    const bool o_first = cand_before(o, v);
    if (low == first_low ? o_first : !o_first) v = o;
}
// Sort the warp's 32 candidates into selection order (lane 0 first).
__device__ __forceinline__ void warp_sort32(Cand &v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
            bitonic_step(v, stride, size == 32 || (lane & size) == 0);
}
// a and b in selection order (one per lane): returns the first 32 of their union, in order.
__device__ __forceinline__ Cand warp_merge32(const Cand &a, const Cand &b) {
    const int lane = threadIdx.x & 31;
    const Cand rb = shfl_cand(b, 31 - lane); // b reversed: a then rb is bitonic
    Cand v = cand_before(rb, a) ? rb : a;    // the 32 first of the 64 (itself bitonic)
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) bitonic_step(v, stride, true);
    return v;
}

// Selection key of a logit a and its remainder b: NaN ranks as -inf, -0 as +0, and a NaN or
// zero remainder as +0.  Never 0 (the key of -inf is above it), so 0 marks "no key yet".
__device__ __forceinline__ unsigned long long cand_key(float a, float b) {
    if (a != a) a = -INFINITY;
    if (a == 0.f) a = 0.f;
    if (b != b || b == 0.f) b = 0.f;
    return ((unsigned long long)float_key(a) << 32) | float_key(b);
}

__device__ __forceinline__ Cand load_cand(const float *lrow, const float *lo_row, int E, int i) {
    Cand c;
    c.key = 0ull; // below every real logit (-inf maps above 0)
    c.id = 0x7fffffff;
    if (i < E) {
        // L2 loads: the logits may come from other CTAs of the same launch
        const float a = __ldcg(lrow + i), b = lo_row ? __ldcg(lo_row + i) : 0.f;
        c.key = cand_key(a, b);
        c.id = i;
    }
    return c;
}

// The gates of a selected list: keys / ids hold the k first candidates in selection order;
// warp 0 forms the softmax over them and writes idx and gate of token t (and, with a
// prediction, counts its hits: P and pred_l as warp 0 read them).  real = false runs the very
// same instructions (a pass that only brings the code into the instruction caches): its idx
// and gate stores are overwritten by the real pass, and it adds zero to the counters.
__device__ __forceinline__ void topk_emit(const unsigned long long *keys, const int *ids, int k, int t,
                                          int32_t *__restrict__ idx, float *__restrict__ gate, int P, int pred_l,
                                          int32_t *__restrict__ pred_count, unsigned long long *__restrict__ stats,
                                          unsigned long long router_bytes, bool real = true) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int my_idx = -1;
        float my_hi = 0.f, my_lo = 0.f;
        if (lane < k) {
            // the selected logit and remainder, as load_cand normalised them, back from the key
            my_idx = ids[lane];
            const unsigned long long key = keys[lane];
            my_hi = key_float((uint32_t)(key >> 32));
            my_lo = key_float((uint32_t)key);
        }
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
            bool hit = false;
            for (int p = 0; p < P && p < 32; ++p) hit |= (__shfl_sync(0xffffffffu, pred_l, p) == my_idx);
            hit = hit && lane < k;
            const unsigned hits = __popc(__ballot_sync(0xffffffffu, hit));
            __syncwarp();
            if (lane == 0) {
                if (P > 0) atomicAdd(stats + kStatPredHits, real ? (unsigned long long)hits : 0ull);
                pred_count[t] = 0;
            }
        }
        if (lane == 0 && stats) {
            atomicAdd(stats + kStatRoutedSlots, real ? (unsigned long long)k : 0ull);
            if (t == 0) atomicAdd(stats + kStatRouter, real ? router_bytes : 0ull);
        }
    }
    __syncthreads();
}

// The warps' lists (each warp's 32 candidates in selection order, one per lane) merged
// pairwise through shared memory: keys / ids (32 entries per warp) end with the first 32 of
// all, in order, at entries 0..31.
__device__ __forceinline__ void merge_warp_lists(const Cand &best, unsigned long long *keys, int *ids) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    keys[warp * 32 + lane] = best.key;
    ids[warp * 32 + lane] = best.id;
    for (int span = 1; span < nw; span <<= 1) {
        __syncthreads();
        if ((warp % (2 * span)) == 0 && warp + span < nw) {
            Cand a, b;
            a.key = keys[warp * 32 + lane];
            a.id = ids[warp * 32 + lane];
            b.key = keys[(warp + span) * 32 + lane];
            b.id = ids[(warp + span) * 32 + lane];
            const Cand m = warp_merge32(a, b);
            __syncwarp();
            keys[warp * 32 + lane] = m.key;
            ids[warp * 32 + lane] = m.id;
        }
    }
    __syncthreads();
}

// Top-k (k <= 32) of one token's logits by the whole CTA: each warp keeps the first 32
// candidates of its 32-wide chunks (sort a chunk, merge), then the warps' lists are merged
// pairwise through shared memory.  keys / ids: scratch of 32 entries per warp.
__device__ __forceinline__ void topk_block(const float *__restrict__ logits,
                                           const float *__restrict__ logits_lo, int E, int k, int t,
                                           int32_t *__restrict__ idx, float *__restrict__ gate,
                                           const int32_t *__restrict__ pred_idx,
                                           int32_t *__restrict__ pred_count, int pred_stride,
                                           unsigned long long *__restrict__ stats,
                                           unsigned long long router_bytes,
                                           unsigned long long *keys, int *ids) {
    const float *lrow = logits + (size_t)t * E;
    const float *lo_row = logits_lo ? logits_lo + (size_t)t * E : nullptr;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    // warp 0 asks for the token's predicted experts now; they arrive during the sort
    int P = 0, pred_l = -1;
    if (warp == 0 && pred_count != nullptr) {
        P = pred_count[t];
        if (lane < pred_stride && lane < P) pred_l = pred_idx[(size_t)t * pred_stride + lane];
    }
    Cand best;
    best.key = 0ull;
    best.id = 0x7fffffff;
    // the warp's chunks c0, c0 + nw * 32, ...: the loads of three chunks in flight at once
    // (the selection is a total order, so the merge order does not change the result)
    constexpr int kAhead = 3;
    for (int c0 = warp * 32; c0 < E; c0 += kAhead * nw * 32) {
        Cand v[kAhead];
#pragma unroll
        for (int q = 0; q < kAhead; ++q) v[q] = load_cand(lrow, lo_row, E, c0 + q * nw * 32 + lane);
#pragma unroll
        for (int q = 0; q < kAhead; ++q)
            if (c0 + q * nw * 32 < E) {
                warp_sort32(v[q]);
                best = warp_merge32(best, v[q]);
            }
    }
    merge_warp_lists(best, keys, ids);
    topk_emit(keys, ids, k, t, idx, gate, P, pred_l, pred_count, stats, router_bytes);
}
} // namespace route
} // namespace wm
