// crc32 of the expert records' payload on the device: the integrity check the page
// "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s" (section "Architecture de streaming
// depuis le disque") puts behind --verify, applied here once when a layer's bank is
// written (waste_moe_pack_records) and when it is opened (waste_moe_create with
// WASTE_FLAG_VERIFY_CRC).
//
// CRC-32 as in IEEE 802.3 / zlib: reflected polynomial 0xEDB88320, register preset to
// all ones, result complemented.  The register update over a byte string is affine in the
// register: R(S, data) = M_len S xor R(0, data), with M_len the GF(2) matrix of "advance
// over len zero bytes".  So the payload is cut into 4 KiB chunks, one thread computes
// R(0, chunk) of each, and one thread per record folds the chunks in order:
// S <- M_4096 S xor R(0, chunk_i) from S = 0xFFFFFFFF; crc = ~S.
#include <vector>

#include "common.cuh"

namespace wm {

namespace {

constexpr uint32_t kCrcPoly = 0xEDB88320u;
constexpr size_t kCrcChunk = 4096;

__host__ __device__ inline uint32_t crc_table_entry(uint32_t i) {
    uint32_t c = i;
    for (int k = 0; k < 8; ++k) c = (c >> 1) ^ (kCrcPoly & (0u - (c & 1u)));
    return c;
}

// R(0, chunk) of every 4 KiB chunk of every record's payload
__global__ void __launch_bounds__(256) crc_chunk_kernel(const uint8_t *__restrict__ records, size_t stride,
                                                        size_t payload_off, size_t n_chunks, int n_records,
                                                        uint32_t *__restrict__ out) {
    __shared__ uint32_t table[256];
    table[threadIdx.x] = crc_table_entry(threadIdx.x);
    __syncthreads();
    const size_t total = n_chunks * (size_t)n_records;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t rec = i / n_chunks, ch = i % n_chunks;
        const uint4 *p = reinterpret_cast<const uint4 *>(records + rec * stride + payload_off + ch * kCrcChunk);
        uint32_t s = 0;
        for (size_t w = 0; w < kCrcChunk / 16; ++w) {
            const uint4 v = __ldg(p + w);
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t x = words[q];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    s = table[(s ^ x) & 0xFFu] ^ (s >> 8);
                    x >>= 8;
                }
            }
        }
        out[i] = s;
    }
}

__device__ inline uint32_t gf2_apply(const uint32_t *cols, uint32_t v) {
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) r ^= cols[i] & (0u - ((v >> i) & 1u));
    return r;
}

struct AdvanceMatrix {
    uint32_t cols[32];
};

// crc of each record from its chunks, in order
__global__ void crc_fold_kernel(const uint32_t *__restrict__ chunk_crc, size_t n_chunks, int n_records,
                                AdvanceMatrix m, uint32_t *__restrict__ out) {
    const int rec = blockIdx.x * blockDim.x + threadIdx.x;
    if (rec >= n_records) return;
    uint32_t s = 0xFFFFFFFFu;
    const uint32_t *c = chunk_crc + (size_t)rec * n_chunks;
    for (size_t i = 0; i < n_chunks; ++i) s = gf2_apply(m.cols, s) ^ c[i];
    out[rec] = ~s;
}

// the folded crc into each record's header field
__global__ void crc_store_kernel(const uint32_t *__restrict__ crc, uint8_t *records, size_t stride, int n_records,
                                 size_t field_off) {
    const int rec = blockIdx.x * blockDim.x + threadIdx.x;
    if (rec < n_records) *reinterpret_cast<uint32_t *>(records + (size_t)rec * stride + field_off) = crc[rec];
}

// GF(2) matrices as 32 columns: column i is the image of bit i.
void gf2_square(const uint32_t *a, uint32_t *out) {
    for (int i = 0; i < 32; ++i) {
        uint32_t r = 0;
        for (int j = 0; j < 32; ++j)
            if ((a[i] >> j) & 1u) r ^= a[j];
        out[i] = r;
    }
}

AdvanceMatrix advance_matrix(size_t bytes) {
    // one zero byte: S -> table[S & 0xFF] ^ (S >> 8), linear in S
    uint32_t m[32], t[32];
    for (int i = 0; i < 32; ++i) {
        const uint32_t s = 1u << i;
        m[i] = crc_table_entry(s & 0xFFu) ^ (s >> 8);
    }
    // bytes is a power of two here: square log2(bytes) times
    size_t n = 1;
    while (n < bytes) {
        gf2_square(m, t);
        for (int i = 0; i < 32; ++i) m[i] = t[i];
        n <<= 1;
    }
    AdvanceMatrix A;
    for (int i = 0; i < 32; ++i) A.cols[i] = m[i];
    return A;
}

} // namespace

cudaError_t launch_payload_crc(const uint8_t *records, size_t stride, int n_records, size_t payload_off,
                               size_t payload_bytes, uint32_t *scratch, uint32_t *crc_out, int num_sms,
                               cudaStream_t s) {
    if (payload_bytes % kCrcChunk) return cudaErrorInvalidValue;
    const size_t n_chunks = payload_bytes / kCrcChunk;
    const size_t total = n_chunks * (size_t)n_records;
    const int grid = (int)std::min<size_t>((total + 255) / 256, (size_t)num_sms * 8);
    crc_chunk_kernel<<<grid, 256, 0, s>>>(records, stride, payload_off, n_chunks, n_records, scratch);
    static const AdvanceMatrix m = advance_matrix(kCrcChunk);
    crc_fold_kernel<<<(n_records + 127) / 128, 128, 0, s>>>(scratch, n_chunks, n_records, m, crc_out);
    return cudaGetLastError();
}

cudaError_t launch_crc_store(const uint32_t *crc, uint8_t *records, size_t stride, int n_records,
                             size_t field_off, cudaStream_t s) {
    crc_store_kernel<<<(n_records + 127) / 128, 128, 0, s>>>(crc, records, stride, n_records, field_off);
    return cudaGetLastError();
}

size_t crc_scratch_words(size_t payload_bytes, int n_records) {
    return payload_bytes / kCrcChunk * (size_t)n_records + (size_t)n_records;
}

} // namespace wm
