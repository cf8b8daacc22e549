// Writing the expert bank: codes in the logical layout -> 4 KiB-aligned
// records (header + gate, up, down sections) in the tiled order the
// table-lookup kernels stream.
//
// Record idea from page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s",
// section "Architecture de streaming depuis le disque": one record per expert,
// aligned to 4 KiB, gate/up/down side by side so one read fetches the expert,
// with magic / expert ID / offset range in a header.
#include "common.cuh"

namespace wm {

namespace {

struct PackArgs {
    MatGeom geom[3];
    const uint8_t *codes[3]; // logical [n][rows][3][nv]
    uint8_t *records;        // record of the first expert
    size_t stride;
    size_t sec_off[3], sec_bytes[3];
    int n;
};

// One thread per output 16-byte chunk; chunks past the tiled area (section
// padding) are zero.  byte q of chunk (sigma, g, s, jj) =
// code[16g + ((jj ^ q) & 15)][s][32 sigma + jj].
__global__ void pack_kernel(const PackArgs P, int m) {
    const MatGeom G = P.geom[m];
    const size_t chunks_per = P.sec_bytes[m] / 16;
    const size_t tiled = G.chunk_bytes() / 16;
    const size_t total = chunks_per * (size_t)P.n;
    const size_t row_bytes = (size_t)kStages * G.nv;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t e = i / chunks_per, c = i % chunks_per;
        uint32_t w[4] = {0, 0, 0, 0};
        if (c < tiled) {
            const int jj = (int)(c % 32);
            const int s = (int)((c / 32) % kStages);
            const size_t gs = c / (32 * kStages);
            const int g = (int)(gs % G.groups);
            const int sigma = (int)(gs / G.groups);
            const int j = sigma * kSegVec + jj;
            if (j < G.nv) {
                const uint8_t *src = P.codes[m] + e * (size_t)G.n_out * row_bytes;
                for (int q = 0; q < 16; ++q) {
                    const int row = g * kGroupRows + ((jj ^ q) & 15);
                    if (row < G.n_out) {
                        const uint32_t b = src[(size_t)row * row_bytes + (size_t)s * G.nv + j];
                        w[q >> 2] |= b << (8 * (q & 3));
                    }
                }
            }
        }
        uint4 *dst = reinterpret_cast<uint4 *>(P.records + e * P.stride + P.sec_off[m]) + c;
        *dst = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void header_kernel(uint8_t *records, size_t stride, int n, waste_record_header hdr,
                              int expert_begin) {
    const int e = blockIdx.x;
    if (e >= n) return;
    uint32_t *page = reinterpret_cast<uint32_t *>(records + (size_t)e * stride);
    for (int i = threadIdx.x; i < (int)(WASTE_RECORD_ALIGN / 4); i += blockDim.x) page[i] = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
        waste_record_header h = hdr;
        h.expert_id = expert_begin + e;
        *reinterpret_cast<waste_record_header *>(page) = h;
    }
}

} // namespace

cudaError_t launch_pack(const MatGeom &gu, const MatGeom &dn, int n_experts,
                        const uint8_t *gate_codes, const uint8_t *up_codes,
                        const uint8_t *down_codes, uint8_t *records, size_t stride,
                        const size_t sec_off[3], cudaStream_t s) {
    PackArgs P;
    P.geom[0] = gu;
    P.geom[1] = gu;
    P.geom[2] = dn;
    P.codes[0] = gate_codes;
    P.codes[1] = up_codes;
    P.codes[2] = down_codes;
    P.records = records;
    P.stride = stride;
    for (int m = 0; m < 3; ++m) {
        P.sec_off[m] = sec_off[m];
        P.sec_bytes[m] = round_up(P.geom[m].chunk_bytes(), WASTE_RECORD_ALIGN);
    }
    P.n = n_experts;
    for (int m = 0; m < 3; ++m) pack_kernel<<<4 * 152, 256, 0, s>>>(P, m);
    return cudaGetLastError();
}

cudaError_t launch_headers(uint8_t *records, size_t stride, int n, const waste_record_header &hdr,
                           int expert_begin, cudaStream_t s) {
    header_kernel<<<n, 256, 0, s>>>(records, stride, n, hdr, expert_begin);
    return cudaGetLastError();
}

} // namespace wm
