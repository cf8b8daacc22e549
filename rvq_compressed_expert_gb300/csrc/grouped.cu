// Batched decode and prefill: the routed (token, expert) slots of a call grouped by
// expert, and every expert that serves enough tokens applied as a dense product on
// the tensor cores.
//
// Pages "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Lecture anticipée
// et prédiction du routeur": one layer of a prefill chunk spans about 550 expert slots,
// so one expert's weights serve many tokens at once.  The weights stay in their
// 3-stage RVQ codes (section "Quantification et exactitude"); here a 128-row tile of
// codes is decoded into shared memory (sum of the three 256-entry codebook rows per
// 8-weight vector) and fed to tcgen05 MMAs with the expert's tokens as the N side.
//
// Kernels, in launch order:
//   group_kernel  per-expert counts, the slots sorted by expert, the chunk list of the
//                 tensor-core experts (<= 128 tokens each) and the list of the slots
//                 left to the lookup kernels (experts with fewer than min_tokens tokens)
//   prep_kernel   the hidden states as fp16 (the B operand)
//   mma_kernel<0> gate and up of every (chunk, 128-row block): two K passes into two
//                 TMEM accumulators, SwiGLU in the epilogue, fp16 result per slot
//   mma_kernel<1> down of every (chunk, 128-row block): y per slot into partial 0
// The lookup kernels serve the listed slots in between, and the combine sums the k
// slots of each token in rank order (one partial for tensor-core slots).
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

// ---------------------------------------------------------------- grouping

constexpr int kGroupThreads = 1024;
constexpr int kExpertsPerThread = kMaxExperts / kGroupThreads; // 4

__global__ void __launch_bounds__(kGroupThreads) group_kernel(const int32_t *__restrict__ idx, int S,
                                                              int E, int min_tokens, Grouping G) {
    __shared__ int cnt[kMaxExperts];
    __shared__ int cur[kMaxExperts];
    __shared__ int2 wsum[kGroupThreads / 32];
    __shared__ int2 total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kGroupThreads) cnt[e] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += kGroupThreads) {
        const int e = idx[s];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive scans over experts of (slots, tensor-core chunks); thread owns experts
    // [4 tid, 4 tid + 4)
    int ls[kExpertsPerThread], lc[kExpertsPerThread];
    int2 mine = make_int2(0, 0);
#pragma unroll
    for (int i = 0; i < kExpertsPerThread; ++i) {
        const int e = kExpertsPerThread * tid + i;
        const int c = e < E ? cnt[e] : 0;
        const int nc = c >= min_tokens ? (c + kGroupTokens - 1) / kGroupTokens : 0;
        ls[i] = mine.x;
        lc[i] = mine.y;
        mine.x += c;
        mine.y += nc;
    }
    int2 inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, inc.x, o);
        const int b = __shfl_up_sync(0xffffffffu, inc.y, o);
        if (lane >= o) {
            inc.x += a;
            inc.y += b;
        }
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int2 v = wsum[lane];
        int2 w = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, w.x, o);
            const int b = __shfl_up_sync(0xffffffffu, w.y, o);
            if (lane >= o) {
                w.x += a;
                w.y += b;
            }
        }
        wsum[lane] = make_int2(w.x - v.x, w.y - v.y);
        if (lane == 31) total = w;
    }
    __syncthreads();
    const int2 base = make_int2(wsum[warp].x + inc.x - mine.x, wsum[warp].y + inc.y - mine.y);
#pragma unroll
    for (int i = 0; i < kExpertsPerThread; ++i) {
        const int e = kExpertsPerThread * tid + i;
        if (e >= E) break;
        const int off = base.x + ls[i];
        G.offs[e] = off;
        cur[e] = off;
        const int c = cnt[e];
        if (c >= min_tokens) {
            const int nc = (c + kGroupTokens - 1) / kGroupTokens;
            for (int j = 0; j < nc; ++j)
                G.chunks[base.y + lc[i] + j] =
                    make_int4(e, off + j * kGroupTokens, min(kGroupTokens, c - j * kGroupTokens), 0);
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

// hidden states (fp32 or bf16) -> fp16, 8 elements per thread
template <bool kBf16>
__global__ void prep_kernel(const void *__restrict__ h, uint16_t *__restrict__ x16, size_t n8) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        float v[8];
        if constexpr (kBf16) {
            const uint4 raw = reinterpret_cast<const uint4 *>(h)[i];
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]));
                v[2 * j] = f.x;
                v[2 * j + 1] = f.y;
            }
        } else {
            const float4 a = reinterpret_cast<const float4 *>(h)[2 * i];
            const float4 b = reinterpret_cast<const float4 *>(h)[2 * i + 1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
        uint4 o;
        uint32_t *ow = &o.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 p = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
            ow[j] = *reinterpret_cast<const uint32_t *>(&p);
        }
        reinterpret_cast<uint4 *>(x16)[i] = o;
    }
}

// ---------------------------------------------------------------- tensor-core kernels

constexpr int kMmaThreads = 512;
constexpr int kBM = 128;              // output rows per item (MMA M)
constexpr int kBK = 64;               // K per chunk: 8 vectors of 8 weights
constexpr int kRing = 4;              // code / activation tile stages
constexpr uint32_t kCopies = 8;       // codebook copies: lane j of a quarter-warp reads copy j
constexpr uint32_t kCbBytes = kStages * kCodes * kCopies * 16;  // 96 KiB of fp16 rows
constexpr uint32_t kABytes = kBM * kBK * 2;                     // 16 KiB
constexpr uint32_t kBBytes = kGroupTokens * kBK * 2;           // 16 KiB
constexpr uint32_t kCodeBytes = 8 * kStages * 8 * 16;          // 8 groups x 3 stages x 8 chunks
constexpr uint32_t kOffCb = 0;
constexpr uint32_t kOffA = kOffCb + kCbBytes;
constexpr uint32_t kOffB = kOffA + 2 * kABytes;
constexpr uint32_t kOffCode = kOffB + kRing * kBBytes;
constexpr uint32_t kOffSlot = kOffCode + kRing * kCodeBytes;
constexpr uint32_t kOffBar = kOffSlot + kGroupTokens * 4;
constexpr uint32_t kOffFlag = kOffBar + 16;
constexpr uint32_t kMmaSmem = kOffFlag + 16;
constexpr uint32_t kTmemCols = 2 * kGroupTokens; // gate and up accumulators
static_assert(kMmaSmem <= 227 * 1024, "shared memory of the tensor-core kernel");

struct MmaArgs {
    const uint8_t *records;
    size_t stride;
    size_t sec[3];
    const float *codebooks;
    MatGeom geom; // the matrix of this kernel (gate/up: f x d, down: d x f)
    int d, f, k, npair;
    const int32_t *sorted;
    const int4 *chunks;
    const int32_t *counts;
    const uint16_t *x16; // [T][d]
    uint16_t *a16;       // [S][f]
    float *part_dn;      // [S][npair][d]
    unsigned long long *stats;
    uint32_t *err;
};

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t half2_bits(float a, float b) {
    const __half2 p = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&p);
}
__device__ __forceinline__ uint32_t hadd2_bits(uint32_t a, uint32_t b) {
    const __half2 r = __hadd2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// One item = (chunk of <= 128 tokens of one expert, 128-row block of the output).  K is
// walked in chunks of 64: the codes of the tile and the chunk's activations arrive by
// cp.async two chunks ahead (4-stage ring), all threads decode the weight tile into an
// A buffer (two of them), one thread issues the four K=16 MMAs and commits them to the
// A buffer's mbarrier.  The MMAs of chunk q run while the weights of chunk q+1 are decoded.
template <bool kDown>
__global__ void __launch_bounds__(kMmaThreads, 1) mma_kernel(const MmaArgs A) {
    extern __shared__ __align__(1024) unsigned char gsm[];
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(gsm);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int *s_slot = reinterpret_cast<int *>(gsm + kOffSlot);
    volatile int *s_flag = reinterpret_cast<volatile int *>(gsm + kOffFlag);
    const uint32_t bar[2] = {sbase + kOffBar, sbase + kOffBar + 8};
    if (tid == 0) {
        tc::mbar_init(bar[0], 1);
        tc::mbar_init(bar[1], 1);
        tc::mbar_init_fence();
        s_flag[0] = 0;
    }
    if (warp == 0) tc::tmem_alloc(sbase + kOffFlag + 4, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gsm + kOffFlag + 4);

    const MatGeom G = A.geom;
    const int nmb = (G.n_out + kBM - 1) / kBM;
    const int KC = (G.n_in + kBK - 1) / kBK;
    const int n_items = A.counts[0] * nmb;
    constexpr int kPasses = kDown ? 1 : 2;
    // decode role: vector column jj of the chunk, row group gq, code bytes 2 qh, 2 qh + 1
    const int jj = lane & 7, gq = warp & 7, qh = (warp >> 3) * 4 + (lane >> 3);
    uint32_t q = 0; // MMA batches committed by this CTA
    bool dead = false;

    for (int item = blockIdx.x; item < n_items && !dead; item += gridDim.x) {
        const int4 ch = A.chunks[item / nmb];
        const int mb = item % nmb;
        const int e = ch.x, start = ch.y, nt = ch.z;
        const int npad = (nt + 15) & ~15;
        const uint32_t idesc = tc::idesc_f16_f32(kBM, npad);
        const uint8_t *rec = A.records + (size_t)e * A.stride;
        __syncthreads(); // the previous item's epilogue is done with s_slot and TMEM
        tc::fence_after_sync();
        if (tid < kGroupTokens) s_slot[tid] = tid < nt ? A.sorted[start + tid] : 0;

        for (int pass = 0; pass < kPasses && !dead; ++pass) {
            const int mat = kDown ? 2 : pass;
            const uint8_t *sec = rec + A.sec[mat];
            // codebook rows of (e, mat) as fp16, kCopies copies side by side
            {
                const float *cb = A.codebooks + ((size_t)e * 3 + mat) * (kStages * kCodes * kVec);
                uint4 *dst = reinterpret_cast<uint4 *>(gsm + kOffCb);
                for (int r = tid; r < kStages * kCodes; r += kMmaThreads) {
                    const float4 lo = __ldg(reinterpret_cast<const float4 *>(cb) + 2 * r);
                    const float4 hi = __ldg(reinterpret_cast<const float4 *>(cb) + 2 * r + 1);
                    const uint4 hv = make_uint4(half2_bits(lo.x, lo.y), half2_bits(lo.z, lo.w),
                                                half2_bits(hi.x, hi.y), half2_bits(hi.z, hi.w));
#pragma unroll
                    for (uint32_t c = 0; c < kCopies; ++c) dst[r * kCopies + c] = hv;
                }
            }
            __syncthreads(); // s_slot (for the loads) and the codebook rows are in place

            auto issue_loads = [&](int kc, uint32_t ring) {
                if (kc < KC) {
                    if (tid < 192) {
                        const int g = tid / 24, s = (tid / 8) % 3, j8 = tid & 7;
                        const int j = kc * 8 + j8, Gg = mb * 8 + g;
                        const bool ok = Gg < G.groups;
                        const uint8_t *src =
                            ok ? sec + (((size_t)(j >> 5) * G.groups + Gg) * kStages + s) * 512 + (j & 31) * 16
                               : sec;
                        cp_async16_zfill(sbase + kOffCode + ring * kCodeBytes + tid * 16, src, ok ? 16u : 0u);
                    }
                    const int npieces = npad * 8;
                    for (int p = tid; p < npieces; p += kMmaThreads) {
                        const int ki = p / npad, n = p - ki * npad;
                        const int kk = kc * kBK + ki * 8;
                        const bool ok = n < nt && kk < G.n_in;
                        const uint16_t *src = A.x16;
                        if (ok) {
                            const int slot = s_slot[n];
                            src = kDown ? A.a16 + (size_t)slot * A.f + kk : A.x16 + (size_t)(slot / A.k) * A.d + kk;
                        }
                        cp_async16_zfill(sbase + kOffB + ring * kBBytes + (n >> 3) * 1024 + ki * 128 + (n & 7) * 16,
                                         src, ok ? 16u : 0u);
                    }
                }
                cp_commit();
            };

            issue_loads(0, q % kRing);
            issue_loads(1, (q + 1) % kRing);
            for (int kc = 0; kc < KC; ++kc, ++q) {
                // ring slot (q + 2) % 4 and A[q & 1] were last read by the MMAs of q - 2,
                // complete since the barrier that closed the previous chunk
                issue_loads(kc + 2, (q + 2) % kRing);
                cp_wait<2>();
                __syncthreads(); // chunk kc's codes and activations are in shared memory
                {
                    const unsigned char *ct = gsm + kOffCode + (q % kRing) * kCodeBytes + (gq * 24 + jj) * 16 + 2 * qh;
                    const uint32_t c0 = *reinterpret_cast<const uint16_t *>(ct);
                    const uint32_t c1 = *reinterpret_cast<const uint16_t *>(ct + 128);
                    const uint32_t c2 = *reinterpret_cast<const uint16_t *>(ct + 256);
                    const int j = kc * 8 + jj, j32 = j & 31;
                    const bool jok = j < G.nv;
                    const uint4 *cbs = reinterpret_cast<const uint4 *>(gsm + kOffCb);
                    unsigned char *abuf = gsm + kOffA + (q & 1) * kABytes;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const int qq = 2 * qh + b;
                        const int rl = 16 * gq + ((j32 ^ qq) & 15);
                        const int row = mb * kBM + rl;
                        const uint4 v0 = cbs[(0 * kCodes + ((c0 >> (8 * b)) & 255)) * kCopies + jj];
                        const uint4 v1 = cbs[(1 * kCodes + ((c1 >> (8 * b)) & 255)) * kCopies + jj];
                        const uint4 v2 = cbs[(2 * kCodes + ((c2 >> (8 * b)) & 255)) * kCopies + jj];
                        uint4 w;
                        w.x = hadd2_bits(hadd2_bits(v0.x, v1.x), v2.x);
                        w.y = hadd2_bits(hadd2_bits(v0.y, v1.y), v2.y);
                        w.z = hadd2_bits(hadd2_bits(v0.z, v1.z), v2.z);
                        w.w = hadd2_bits(hadd2_bits(v0.w, v1.w), v2.w);
                        if (!jok || row >= G.n_out) w = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(abuf + (rl >> 3) * 1024 + jj * 128 + (rl & 7) * 16) = w;
                    }
                }
                tc::fence_proxy_async();
                if (tid == 0 && q >= 1 && !tc::mbar_wait(bar[(q - 1) & 1], ((q - 1) >> 1) & 1)) s_flag[0] = 1;
                __syncthreads(); // tile decoded; the MMAs of q - 1 are complete
                if (s_flag[0]) {
                    dead = true;
                    break;
                }
                if (tid == 0) {
                    tc::fence_after_sync();
                    const uint32_t a_addr = sbase + kOffA + (q & 1) * kABytes;
                    const uint32_t b_addr = sbase + kOffB + (q % kRing) * kBBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc::mma_f16(tmem + pass * kGroupTokens, tc::smem_desc(a_addr + kk * 256, 128, 1024),
                                    tc::smem_desc(b_addr + kk * 256, 128, 1024), idesc, (kc | kk) != 0);
                    tc::mma_commit(bar[q & 1]);
                }
            }
        }
        if (dead) break;
        // the item's last MMAs
        if (tid == 0 && !tc::mbar_wait(bar[(q - 1) & 1], ((q - 1) >> 1) & 1)) s_flag[0] = 1;
        __syncthreads();
        if (s_flag[0]) {
            dead = true;
            break;
        }
        tc::fence_after_sync();
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. +32 (its output rows) and
        // column blocks of 16 starting at 16 (w / 4), every 64
        {
            const int lq = warp & 3;
            const int rl = lq * 32 + lane, row = mb * kBM + rl;
            const uint32_t lane_addr = tmem + ((uint32_t)(lq * 32) << 16);
            for (int c0 = (warp >> 2) * 16; c0 < npad; c0 += 64) {
                float z[16];
                tc::tmem_ld16(lane_addr + c0, z);
                if constexpr (!kDown) {
                    float u[16];
                    tc::tmem_ld16(lane_addr + kGroupTokens + c0, u);
                    if (row < G.n_out) {
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            if (c0 + n < nt) {
                                const float a = z[n] / (1.0f + expf(-z[n])) * u[n];
                                const __half ha = __float2half_rn(a);
                                A.a16[(size_t)s_slot[c0 + n] * A.f + row] = *reinterpret_cast<const uint16_t *>(&ha);
                            }
                    }
                } else {
                    if (row < G.n_out) {
#pragma unroll
                        for (int n = 0; n < 16; ++n)
                            if (c0 + n < nt) A.part_dn[(size_t)s_slot[c0 + n] * A.npair * A.d + row] = z[n];
                    }
                }
            }
        }
        tc::fence_before_sync();
        if (tid == 0 && A.stats) {
            const int rows = min(G.n_out - mb * kBM, kBM);
            atomicAdd(A.stats + kStatDemandCode,
                      (unsigned long long)kPasses * rows * G.nv * kStages);
            if (mb == 0)
                atomicAdd(A.stats + kStatCodebook,
                          (unsigned long long)kPasses * kStages * kCodes * kVec * sizeof(float));
        }
    }
    cp_wait<0>();
    if (dead) {
        // give the MMAs in flight a bounded chance to finish before TMEM is released
        if (tid == 0) {
            if (q >= 1) tc::mbar_wait(bar[(q - 1) & 1], ((q - 1) >> 1) & 1);
            atomicOr(A.err, kErrTimeout);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kDown>
cudaError_t launch_mma(const MmaArgs &A, int num_sms, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(mma_kernel<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kMmaSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    mma_kernel<kDown><<<num_sms, kMmaThreads, kMmaSmem, s>>>(A);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_grouped_forward(const LayerView &L, const Workspace &W, const void *h, int T,
                                   const int32_t *idx, const float *gate, float *out, int mode,
                                   int min_tokens, bool reconstruct, int num_sms, cudaStream_t s,
                                   Timing *tm) {
    const Grouping &G = W.grp;
    const int S = T * L.k;
    if (tm) cudaEventRecord(tm->ev[0], s);
    group_kernel<<<1, kGroupThreads, 0, s>>>(idx, S, L.E, min_tokens < 1 ? 1 : min_tokens, G);
    const size_t n8 = (size_t)T * L.d / 8;
    const int pgrid = (int)((n8 + 255) / 256 < (size_t)(num_sms * 8) ? (n8 + 255) / 256 : (size_t)(num_sms * 8));
    if (L.act_bf16)
        prep_kernel<true><<<pgrid, 256, 0, s>>>(h, G.x16, n8);
    else
        prep_kernel<false><<<pgrid, 256, 0, s>>>(h, G.x16, n8);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    MmaArgs A;
    A.records = L.records;
    A.stride = L.stride;
    for (int m = 0; m < 3; ++m) A.sec[m] = L.sec_off[m];
    A.codebooks = L.codebooks;
    A.d = L.d;
    A.f = L.f;
    A.k = L.k;
    A.npair = (L.dn.nseg + 1) / 2;
    A.sorted = G.sorted;
    A.chunks = G.chunks;
    A.counts = G.counts;
    A.x16 = G.x16;
    A.a16 = G.a16;
    A.part_dn = W.part_dn;
    A.stats = W.stats;
    A.err = W.err;

    // gate/up: lookup slots, then the tensor-core chunks
    e = launch_lut_listed(L, W, h, T, idx, G.lut_slots, G.counts + 1, false, reconstruct, num_sms, s);
    if (e != cudaSuccess) return e;
    A.geom = L.gu;
    e = launch_mma<false>(A, num_sms, s);
    if (e != cudaSuccess) return e;
    if (tm) cudaEventRecord(tm->ev[1], s);
    // down
    e = launch_lut_listed(L, W, h, T, idx, G.lut_slots, G.counts + 1, true, reconstruct, num_sms, s);
    if (e != cudaSuccess) return e;
    A.geom = L.dn;
    e = launch_mma<true>(A, num_sms, s);
    if (e != cudaSuccess) return e;
    if (tm) cudaEventRecord(tm->ev[2], s);
    e = launch_combine(L, W, h, T, idx, gate, out, mode, G.one_part, s);
    if (e != cudaSuccess) return e;
    if (tm) {
        cudaEventRecord(tm->ev[3], s);
        tm->n = 4;
    }
    return cudaSuccess;
}

} // namespace wm
