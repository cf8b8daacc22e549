// waste_moe_forward_noalloc: the expert forward (gate/up, down, combine) without a
// handle and without any allocation.
//
// The table-lookup kernels keep per-segment partial sums in global scratch.  A handle
// gets that scratch from cudaMalloc at create time; some callers cannot allocate
// device memory at all -- a host that only receives device pointers from an engine
// owning every byte of HBM, or code that runs where allocation is forbidden.  For them
// the scratch lives in a fixed array in this library's device image instead.
#include "common.cuh"

#include <mutex>

using namespace wm;

namespace {

// Scratch for the no-allocation forward: 8 MiB, resident on every device that loads
// the library until the process exits.  Layout: [256 B: device error word][gate/up
// partials][down partials].
constexpr size_t kStaticScratchBytes = 8u << 20;

__device__ __align__(256) unsigned char g_forward_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

int fail_na(int code, const char *msg) {
    set_last_error(msg);
    return code;
}

// Device address of the scratch array on the current device, looked up once per device.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_forward_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" {

int waste_moe_forward_noalloc(const waste_moe_config *cfg, const uint8_t *d_records,
                              size_t record_stride, const float *d_codebooks, const void *d_h,
                              int32_t T, const int32_t *d_idx, const float *d_gate,
                              float *d_out, int32_t mode, waste_stream_t stream) {
    const NvtxRange nvtx_range(__func__);
    if (!cfg || cfg->abi_version != WASTE_MOE_ABI_VERSION)
        return fail_na(WASTE_EINVAL, "config is NULL or of another ABI version");
    if (cfg->d <= 0 || cfg->d % kVec || cfg->f <= 0 || cfg->f % kVec || cfg->n_experts < 1 ||
        cfg->n_experts > kMaxExperts || cfg->top_k < 1 || cfg->top_k > cfg->n_experts ||
        cfg->top_k > kMaxTopK || (cfg->act_dtype != WASTE_ACT_F32 && cfg->act_dtype != WASTE_ACT_BF16))
        return fail_na(WASTE_EINVAL, "bad shapes in config");
    if (T < 0) return fail_na(WASTE_EINVAL, "T < 0");
    if (mode < 0 || mode > 2 || (mode == 2 && cfg->act_dtype != WASTE_ACT_F32))
        return fail_na(WASTE_EINVAL, "bad mode");
    if (T == 0) return WASTE_OK;
    if (!d_records || !d_codebooks || !d_h || !d_idx || !d_gate || !d_out)
        return fail_na(WASTE_EINVAL, "NULL pointer");
    if ((uintptr_t)d_records % WASTE_RECORD_ALIGN || (uintptr_t)d_h % 16 ||
        (uintptr_t)d_codebooks % 16)
        return fail_na(WASTE_EINVAL, "misaligned records, codebooks or hidden states");

    LayerView L;
    L.gu = mat_geom(cfg->f, cfg->d);
    L.dn = mat_geom(cfg->d, cfg->f);
    size_t sec[3];
    sec[0] = round_up(L.gu.chunk_bytes(), WASTE_RECORD_ALIGN);
    sec[1] = sec[0];
    sec[2] = round_up(L.dn.chunk_bytes(), WASTE_RECORD_ALIGN);
    L.sec_off[0] = WASTE_RECORD_ALIGN;
    L.sec_off[1] = L.sec_off[0] + sec[0];
    L.sec_off[2] = L.sec_off[1] + sec[1];
    if (record_stride < L.sec_off[2] + sec[2] || record_stride % WASTE_RECORD_ALIGN)
        return fail_na(WASTE_EINVAL, "record stride too small or not a multiple of 4096");

    // scratch demand of this call against the fixed array
    const size_t slots = (size_t)T * (size_t)cfg->top_k;
    const size_t npair = (size_t)down_parts(L);
    const size_t gu_bytes = round_up(slots * (size_t)((L.gu.nseg + 1) / 2) * 2 * (size_t)cfg->f * 4, 256);
    const size_t dn_bytes = round_up(slots * npair * (size_t)cfg->d * 4, 256);
    if (256 + gu_bytes + dn_bytes > kStaticScratchBytes)
        return fail_na(WASTE_EINVAL,
                       "T * top_k slots need more partial-sum scratch than the fixed 8 MiB "
                       "array holds; use waste_moe_forward with a handle");

    void *base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) return fail_na(WASTE_ECUDA, cudaGetErrorString(e));

    L.router_w = nullptr;
    L.router_b = nullptr;
    L.records = d_records;
    L.slot_map = nullptr;
    L.stride = record_stride;
    L.codebooks = d_codebooks;
    L.d = cfg->d;
    L.f = cfg->f;
    L.E = cfg->n_experts;
    L.k = cfg->top_k;
    L.act_bf16 = cfg->act_dtype == WASTE_ACT_BF16;

    Workspace W = {};
    unsigned char *b = static_cast<unsigned char *>(base);
    W.err = reinterpret_cast<uint32_t *>(b);
    W.part_gu = reinterpret_cast<float *>(b + 256);
    W.part_dn = reinterpret_cast<float *>(b + 256 + gu_bytes);
    W.stats = nullptr;
    e = launch_lut_forward(L, W, d_h, T, d_idx, d_gate, d_out, mode,
                           (cfg->flags & WASTE_FLAG_K2_RECONSTRUCT) != 0, device_sm_count(),
                           reinterpret_cast<cudaStream_t>(stream), nullptr);
    if (e != cudaSuccess) return fail_na(WASTE_ECUDA, cudaGetErrorString(e));
    set_last_error("");
    return WASTE_OK;
}

} // extern "C"
