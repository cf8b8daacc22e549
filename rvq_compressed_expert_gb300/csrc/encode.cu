// RVQ encoder: codes and codebooks of a dense matrix, the step before the path.
//
// Page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section "Quantification et
// exactitude": experts are stored as 3 residual stages of 256 eight-dimensional vectors; the
// converter that writes them is named, its training is not.  This is greedy residual k-means:
// per stage, centroids start on given vectors of the residual, `iters` Lloyd rounds move each
// used centroid to the mean of its members, a last assignment gives the stage's codes and the
// residual drops the chosen centroid.
//
// Exactness: the nearest centroid is the least sum over v of (x_v - c_v)^2 taken in fp32 in
// order v = 0..7 with one fused multiply-add per term, ties to the lower index, so a code is
// the same integer any fp32 implementation of that rule would pick.  Centroid sums are carried
// in fixed point (round(x * 2^40) as int64), exact in any order, so shared-memory and global
// atomics give the same means on every run.
//
// Kernels: an assignment pass (persistent CTAs of 256 threads, four vectors per thread, the 256
// centroids in shared memory; it either adds each vector to its centroid's sums in shared
// memory, flushed once per CTA, or applies the stage: residual update, code, squared error),
// a mean kernel, a centroid-init gather and an input check.  Bound: fp32 issue (16 operations
// per vector and centroid).
#include <new>

#include "common.cuh"

namespace wm {

namespace {

constexpr int kK = 256;
constexpr int kV = 8;
constexpr int kAssignThreads = 256;
constexpr int kPerThread = 4;
constexpr double kFix = 1099511627776.0; // 2^40

struct EncScratch {
    float *R;                  // [n][8] residual
    unsigned long long *sums;  // [256][8] fixed-point sums (two's complement)
    unsigned long long *cnt;   // [256]
    uint32_t *flag;            // input check
};

__global__ void check_kernel(const float *__restrict__ W, size_t n_elems, const int32_t *__restrict__ init,
                             int n_init, size_t n_vec, uint32_t *flag) {
    const size_t step = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_elems; i += step)
        if (!(fabsf(W[i]) < 4194304.0f)) atomicOr(flag, 1u);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)n_init; i += step)
        if (init[i] < 0 || (size_t)init[i] >= n_vec) atomicOr(flag, 2u);
}

__global__ void init_kernel(const float *__restrict__ R, const int32_t *__restrict__ init, float *__restrict__ C) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < kK * kV) C[t] = R[(size_t)init[t / kV] * kV + (t % kV)];
}

__global__ void means_kernel(const unsigned long long *__restrict__ sums, const unsigned long long *__restrict__ cnt,
                             float *__restrict__ C) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= kK * kV) return;
    const unsigned long long n = cnt[t / kV];
    if (n == 0) return; // an empty centroid keeps its value
    const long long s = (long long)sums[t];
    C[t] = (float)(((double)s / (double)n) * (1.0 / kFix));
}

__device__ __forceinline__ void load_vec(const float *p, float x[kV]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0];
    const float4 b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// kApply = false: add each vector to its nearest centroid's sums.  kApply = true: the stage's
// codes into codes[r][stage][j], R -= C[code], and the squared residual into *err.
template <bool kApply>
__global__ void __launch_bounds__(kAssignThreads) assign_kernel(float *__restrict__ R, size_t n, const float *__restrict__ Cg,
                                                                unsigned long long *__restrict__ sums,
                                                                unsigned long long *__restrict__ cnt, uint8_t *__restrict__ codes,
                                                                int nv, int stage, double *__restrict__ err) {
    __shared__ __align__(16) float C[kK * kV];
    __shared__ unsigned long long s_sum[kApply ? 1 : kK * kV];
    __shared__ unsigned long long s_cnt[kApply ? 1 : kK];
    __shared__ double s_err[kAssignThreads / 32];
    for (int i = threadIdx.x; i < kK * kV; i += kAssignThreads) C[i] = Cg[i];
    if constexpr (!kApply) {
        for (int i = threadIdx.x; i < kK * kV; i += kAssignThreads) s_sum[i] = 0ull;
        for (int i = threadIdx.x; i < kK; i += kAssignThreads) s_cnt[i] = 0ull;
    }
    __syncthreads();
    double e = 0.0;
    const size_t per_cta = (size_t)kAssignThreads * kPerThread;
    for (size_t base = (size_t)blockIdx.x * per_cta; base < n; base += (size_t)gridDim.x * per_cta) {
        float x[kPerThread][kV];
        size_t vi[kPerThread];
        bool ok[kPerThread];
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            vi[u] = base + (size_t)u * kAssignThreads + threadIdx.x;
            ok[u] = vi[u] < n;
            if (ok[u]) load_vec(R + vi[u] * kV, x[u]);
            else
#pragma unroll
                for (int v = 0; v < kV; ++v) x[u][v] = 0.f;
        }
        float bd[kPerThread];
        int best[kPerThread];
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            bd[u] = __int_as_float(0x7f800000); // +inf
            best[u] = 0;
        }
#pragma unroll 4
        for (int c = 0; c < kK; ++c) {
            const float4 ca = reinterpret_cast<const float4 *>(C)[2 * c];
            const float4 cb = reinterpret_cast<const float4 *>(C)[2 * c + 1];
            const float cv[kV] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
            for (int u = 0; u < kPerThread; ++u) {
                float d = 0.f;
#pragma unroll
                for (int v = 0; v < kV; ++v) {
                    const float t = __fsub_rn(x[u][v], cv[v]);
                    d = __fmaf_rn(t, t, d);
                }
                if (d < bd[u]) {
                    bd[u] = d;
                    best[u] = c;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            if (!ok[u]) continue;
            const int c = best[u];
            if constexpr (kApply) {
                float r[kV];
#pragma unroll
                for (int v = 0; v < kV; ++v) {
                    r[v] = __fsub_rn(x[u][v], C[c * kV + v]);
                    e += (double)r[v] * (double)r[v];
                }
                float4 *dst = reinterpret_cast<float4 *>(R + vi[u] * kV);
                dst[0] = make_float4(r[0], r[1], r[2], r[3]);
                dst[1] = make_float4(r[4], r[5], r[6], r[7]);
                const size_t row = vi[u] / (size_t)nv, j = vi[u] % (size_t)nv;
                codes[(row * 3 + (size_t)stage) * (size_t)nv + j] = (uint8_t)c;
            } else {
                atomicAdd(&s_cnt[c], 1ull);
#pragma unroll
                for (int v = 0; v < kV; ++v)
                    atomicAdd(&s_sum[c * kV + v], (unsigned long long)__double2ll_rn((double)x[u][v] * kFix));
            }
        }
    }
    if constexpr (kApply) {
        // the block's squared error: warp sums, then one add per block
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
        if ((threadIdx.x & 31) == 0) s_err[threadIdx.x >> 5] = e;
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int w = 0; w < kAssignThreads / 32; ++w) t += s_err[w];
            atomicAdd(err, t);
        }
    } else {
        __syncthreads();
        for (int i = threadIdx.x; i < kK * kV; i += kAssignThreads)
            if (s_sum[i]) atomicAdd(&sums[i], s_sum[i]);
        for (int i = threadIdx.x; i < kK; i += kAssignThreads)
            if (s_cnt[i]) atomicAdd(&cnt[i], s_cnt[i]);
    }
}

// CTAs of an assignment pass: at most four per SM (all resident), and as many rounds for
// each CTA as the largest of them needs, so the last round is not a partial one.
int assign_grid(size_t n, int num_sms) {
    const size_t per_cta = (size_t)kAssignThreads * kPerThread;
    const size_t need = (n + per_cta - 1) / per_cta;
    const size_t cap = (size_t)num_sms * 4;
    if (need <= cap) return (int)(need ? need : 1);
    const size_t rounds = (need + cap - 1) / cap;
    return (int)((need + rounds - 1) / rounds);
}

int enc_fail(int code, const char *msg) {
    set_last_error(msg);
    return code;
}

} // namespace

} // namespace wm

using namespace wm;

namespace {

// Validates the shapes, allocates the scratch, copies W into the residual and checks the
// input on the device (synchronous).  init may be null (encode).
int enc_begin(const float *d_w, int32_t rows, int32_t cols, const int32_t *d_init, cudaStream_t s, EncScratch &S,
              size_t &n) {
    S = EncScratch{};
    if (!d_w || rows < 1 || cols < 8 || cols % kV) return enc_fail(WASTE_EINVAL, "need W, rows >= 1, cols a multiple of 8");
    n = (size_t)rows * (size_t)(cols / kV);
    void *mem = nullptr;
    const size_t rbytes = round_up(n * kV * 4, 256);
    cudaError_t e = cudaMalloc(&mem, rbytes + kK * kV * 8 + kK * 8 + 256);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return enc_fail(WASTE_ENOMEM, "encoder scratch");
    }
    char *b = static_cast<char *>(mem);
    S.R = reinterpret_cast<float *>(b);
    S.sums = reinterpret_cast<unsigned long long *>(b + rbytes);
    S.cnt = S.sums + kK * kV;
    S.flag = reinterpret_cast<uint32_t *>(S.cnt + kK);
    e = cudaMemsetAsync(S.flag, 0, 4, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(S.R, d_w, n * kV * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) {
        check_kernel<<<device_sm_count() * 2, 256, 0, s>>>(d_w, n * kV, d_init, d_init ? 3 * kK : 0, n, S.flag);
        e = cudaGetLastError();
    }
    uint32_t flag = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&flag, S.flag, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaFree(mem);
        S.R = nullptr;
        return enc_fail(WASTE_ECUDA, cudaGetErrorString(e));
    }
    if (flag) {
        cudaFree(mem);
        S.R = nullptr;
        return enc_fail(WASTE_EINVAL, flag & 1u ? "a weight is not finite or has |w| >= 2^22"
                                                : "an init index is outside the matrix's vectors");
    }
    return WASTE_OK;
}

int enc_end(EncScratch &S, cudaStream_t s, cudaError_t e) {
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(S.R);
    if (e != cudaSuccess) return enc_fail(WASTE_ECUDA, cudaGetErrorString(e));
    set_last_error("");
    return WASTE_OK;
}

// The stage's final assignment: codes, residual update, squared error.
cudaError_t apply_stage(EncScratch &S, size_t n, const float *C, uint8_t *codes, int nv, int stage, double *err,
                        int num_sms, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(err + stage, 0, 8, s);
    if (e != cudaSuccess) return e;
    assign_kernel<true><<<assign_grid(n, num_sms), kAssignThreads, 0, s>>>(S.R, n, C, nullptr, nullptr, codes, nv,
                                                                         stage, err + stage);
    return cudaGetLastError();
}

} // namespace

extern "C" {

int waste_rvq_train(const float *d_w, int32_t rows, int32_t cols, const int32_t *d_init, int32_t iters,
                    float *d_codebooks, uint8_t *d_codes, double *d_err, waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    if (!d_init || !d_codebooks || !d_codes || !d_err || iters < 0)
        return enc_fail(WASTE_EINVAL, "NULL init, codebooks, codes or err, or iters < 0");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    EncScratch S;
    size_t n = 0;
    int rc = enc_begin(d_w, rows, cols, d_init, s, S, n);
    if (rc) return rc;
    const int nv = cols / kV, sms = device_sm_count();
    cudaError_t e = cudaSuccess;
    for (int st = 0; st < 3 && e == cudaSuccess; ++st) {
        float *C = d_codebooks + (size_t)st * kK * kV;
        init_kernel<<<kK * kV / 256, 256, 0, s>>>(S.R, d_init + st * kK, C);
        e = cudaGetLastError();
        for (int it = 0; it < iters && e == cudaSuccess; ++it) {
            e = cudaMemsetAsync(S.sums, 0, (kK * kV + kK) * 8, s);
            if (e != cudaSuccess) break;
            assign_kernel<false><<<assign_grid(n, sms), kAssignThreads, 0, s>>>(S.R, n, C, S.sums, S.cnt, nullptr, nv,
                                                                              st, nullptr);
            means_kernel<<<kK * kV / 256, 256, 0, s>>>(S.sums, S.cnt, C);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) e = apply_stage(S, n, C, d_codes, nv, st, d_err, sms, s);
    }
    return enc_end(S, s, e);
}

int waste_rvq_encode(const float *d_w, int32_t rows, int32_t cols, const float *d_codebooks, uint8_t *d_codes,
                     double *d_err, waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    if (!d_codebooks || !d_codes || !d_err) return enc_fail(WASTE_EINVAL, "NULL codebooks, codes or err");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    EncScratch S;
    size_t n = 0;
    int rc = enc_begin(d_w, rows, cols, nullptr, s, S, n);
    if (rc) return rc;
    const int nv = cols / kV, sms = device_sm_count();
    cudaError_t e = cudaSuccess;
    for (int st = 0; st < 3 && e == cudaSuccess; ++st)
        e = apply_stage(S, n, d_codebooks + (size_t)st * kK * kV, d_codes, nv, st, d_err, sms, s);
    return enc_end(S, s, e);
}

} // extern "C"
