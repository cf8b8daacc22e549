// crc32 of the expert records' payload on the device: the integrity check the page
// "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s" (section "Architecture de streaming
// depuis le disque") puts behind --verify, applied here once when a layer's bank is
// written (waste_moe_pack_records) and when it is opened (waste_moe_create with
// WASTE_FLAG_VERIFY_CRC).
//
// CRC-32 as in IEEE 802.3 / zlib: reflected polynomial 0xEDB88320, register preset to
// all ones, result complemented.  The register update over a byte string is affine in the
// register: R(S, data) = M_len S xor R(0, data), with M_len the GF(2) matrix of "advance
// over len zero bytes", and R(0, .) ignores leading zero bytes.  So the payload is cut into
// 4 KiB chunks and a thread computes R(0, chunk) of each, four bytes per dependent step
// (four 256-entry tables); then one warp per record folds its chunks: each lane folds an
// equal run of chunks (the record padded in front with zero chunks to 32 equal runs), the
// lanes combine in a shuffle tree, R(0, A||B) = M_len(B) R(0, A) xor R(0, B), and
// crc = ~(M_payload 0xFFFFFFFF xor R(0, payload)).
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

// One chunk per warp, read coalesced: lane l takes the 16-byte pieces l, l + 32, ..., l + 224.
// Piece p's contribution to R(0, chunk) is M_{16 (255 - p)} R(0, piece) = M_{512 (7 - j)}
// M_{16 (31 - l)} R(0, piece) for p = 32 j + l, so a lane folds its pieces with the advance
// over 512 bytes (four byte tables of that matrix) and the lanes combine in a shuffle tree,
// R(0, A||B) = M_{16 |B|} R(0, A) xor R(0, B).  R(0, piece) four bytes per step: for each
// 32-bit little-endian word w, x = S ^ w and S = T3[x & 255] ^ T2[x >> 8 & 255] ^
// T1[x >> 16 & 255] ^ T0[x >> 24], with T0 the byte table and T_k[i] = (T_{k-1}[i] >> 8) ^
// T0[T_{k-1}[i] & 255] (the same update as four byte steps).
struct ChunkArgs {
    uint32_t adv512[32];   // advance over 512 zero bytes
    uint32_t tree[5][32];  // advance over 16 * 2^k zero bytes
};

__device__ __forceinline__ uint32_t gf2_cols(const uint32_t *cols, uint32_t v) {
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) r ^= cols[i] & (0u - ((v >> i) & 1u));
    return r;
}

__global__ void __launch_bounds__(256) crc_chunk_kernel(const uint8_t *__restrict__ records, size_t stride,
                                                        size_t payload_off, size_t n_chunks, int n_records,
                                                        const ChunkArgs C, uint32_t *__restrict__ out) {
    __shared__ uint32_t table[4][256];
    __shared__ uint32_t adv[4][256];
    table[0][threadIdx.x] = crc_table_entry(threadIdx.x);
#pragma unroll
    for (int k = 0; k < 4; ++k) adv[k][threadIdx.x] = gf2_cols(C.adv512, threadIdx.x << (8 * k));
    __syncthreads();
#pragma unroll
    for (int k = 1; k < 4; ++k) {
        const uint32_t t = table[k - 1][threadIdx.x];
        table[k][threadIdx.x] = (t >> 8) ^ table[0][t & 0xFFu];
        __syncthreads();
    }
    const int lane = threadIdx.x & 31;
    const size_t total = n_chunks * (size_t)n_records;
    const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
    for (size_t i = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < total; i += warps) {
        const size_t rec = i / n_chunks, ch = i % n_chunks;
        const uint4 *p = reinterpret_cast<const uint4 *>(records + rec * stride + payload_off + ch * kCrcChunk);
        uint4 v[kCrcChunk / 512];
#pragma unroll
        for (int j = 0; j < (int)(kCrcChunk / 512); ++j) v[j] = __ldg(p + 32 * j + lane); // all in flight
        uint32_t acc = 0;
#pragma unroll
        for (int j = 0; j < (int)(kCrcChunk / 512); ++j) {
            const uint32_t words[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t s = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t x = s ^ words[q];
                s = table[3][x & 0xFFu] ^ table[2][(x >> 8) & 0xFFu] ^ table[1][(x >> 16) & 0xFFu] ^ table[0][x >> 24];
            }
            acc = adv[0][acc & 0xFFu] ^ adv[1][(acc >> 8) & 0xFFu] ^ adv[2][(acc >> 16) & 0xFFu] ^ adv[3][acc >> 24] ^ s;
        }
#pragma unroll
        for (int k = 0; k < 5; ++k) {
            const uint32_t t = __shfl_down_sync(0xffffffffu, acc, 1 << k);
            const uint32_t m = gf2_cols(C.tree[k], acc) ^ t;
            if ((lane & ((2 << k) - 1)) == 0) acc = m;
        }
        if (lane == 0) out[i] = acc;
    }
}

__host__ __device__ inline uint32_t gf2_apply(const uint32_t *cols, uint32_t v) {
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) r ^= cols[i] & (0u - ((v >> i) & 1u));
    return r;
}

// Matrices of one fold: advance over one chunk, over 2^k lane runs (k = 0..4), and the
// preset register advanced over the whole payload.
struct FoldArgs {
    uint32_t chunk[32];
    uint32_t tree[5][32];
    uint32_t preset;
    int run;  // chunks per lane
    int pad;  // zero chunks in front of the record
};

// crc of each record from its chunks: one warp per record
__global__ void __launch_bounds__(128) crc_fold_kernel(const uint32_t *__restrict__ chunk_crc, size_t n_chunks,
                                                       int n_records, const FoldArgs F, uint32_t *__restrict__ out) {
    const int rec = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (rec >= n_records) return; // whole warps leave together
    const uint32_t *c = chunk_crc + (size_t)rec * n_chunks;
    uint32_t s = 0;
    const long long first = (long long)lane * F.run - F.pad;
    for (long long i = first < 0 ? 0 : first; i < first + F.run; ++i) s = gf2_apply(F.chunk, s) ^ c[i];
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, s, 1 << k);
        const uint32_t m = gf2_apply(F.tree[k], s) ^ t;
        if ((lane & ((2 << k) - 1)) == 0) s = m;
    }
    if (lane == 0) out[rec] = ~(F.preset ^ s);
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

// a * b (apply b, then a)
void gf2_mul(const uint32_t *a, const uint32_t *b, uint32_t *out) {
    uint32_t r[32];
    for (int i = 0; i < 32; ++i) r[i] = gf2_apply(a, b[i]);
    for (int i = 0; i < 32; ++i) out[i] = r[i];
}

// m^n by squaring
void gf2_pow(const uint32_t *m, size_t n, uint32_t *out) {
    uint32_t r[32], b[32], t[32];
    for (int i = 0; i < 32; ++i) {
        r[i] = 1u << i;
        b[i] = m[i];
    }
    while (n) {
        if (n & 1) gf2_mul(b, r, r);
        gf2_square(b, t);
        for (int i = 0; i < 32; ++i) b[i] = t[i];
        n >>= 1;
    }
    for (int i = 0; i < 32; ++i) out[i] = r[i];
}

void byte_matrix(uint32_t *m) {
    // one zero byte: S -> table[S & 0xFF] ^ (S >> 8), linear in S
    for (int i = 0; i < 32; ++i) {
        const uint32_t s = 1u << i;
        m[i] = crc_table_entry(s & 0xFFu) ^ (s >> 8);
    }
}

ChunkArgs chunk_args() {
    uint32_t byte[32];
    byte_matrix(byte);
    ChunkArgs C;
    gf2_pow(byte, 512, C.adv512);
    for (int k = 0; k < 5; ++k) gf2_pow(byte, (size_t)16 << k, C.tree[k]);
    return C;
}

FoldArgs fold_args(size_t n_chunks) {
    // one zero byte: S -> table[S & 0xFF] ^ (S >> 8), linear in S
    uint32_t byte[32];
    for (int i = 0; i < 32; ++i) {
        const uint32_t s = 1u << i;
        byte[i] = crc_table_entry(s & 0xFFu) ^ (s >> 8);
    }
    FoldArgs F;
    gf2_pow(byte, kCrcChunk, F.chunk);
    F.run = (int)((n_chunks + 31) / 32);
    F.pad = (int)(32 * (size_t)F.run - n_chunks);
    for (int k = 0; k < 5; ++k) gf2_pow(F.chunk, (size_t)F.run << k, F.tree[k]);
    uint32_t all[32];
    gf2_pow(F.chunk, n_chunks, all);
    F.preset = gf2_apply(all, 0xFFFFFFFFu);
    return F;
}

} // namespace

cudaError_t launch_payload_crc(const uint8_t *records, size_t stride, int n_records, size_t payload_off,
                               size_t payload_bytes, uint32_t *scratch, uint32_t *crc_out, int num_sms,
                               cudaStream_t s) {
    if (payload_bytes % kCrcChunk) return cudaErrorInvalidValue;
    const size_t n_chunks = payload_bytes / kCrcChunk;
    const size_t total = n_chunks * (size_t)n_records;
    const int grid = (int)std::min<size_t>((total + 7) / 8, (size_t)num_sms * 8); // 8 chunks (warps) per CTA
    static const ChunkArgs C = chunk_args();
    crc_chunk_kernel<<<grid, 256, 0, s>>>(records, stride, payload_off, n_chunks, n_records, C, scratch);
    const FoldArgs F = fold_args(n_chunks);
    crc_fold_kernel<<<(n_records + 3) / 4, 128, 0, s>>>(scratch, n_chunks, n_records, F, crc_out);
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
