// Device-side pieces of the table-lookup expert kernels, shared by the per-phase
// kernels (lut_gemv.cu) and the fused decode-step kernel (fused.cu).
#pragma once

#include "common.cuh"
#include "tc_dev.cuh"

#include <type_traits>


namespace wm {
namespace lut {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kTabStage = 65536;             // bytes per stage: 256 codes x 256 B
constexpr int kTabBytes = kStages * kTabStage; // 192 KiB
constexpr int kXsFloats = 512;               // down input staging (64 vectors x 8)
constexpr int kCbFloats = kStages * kCodes * kVec; // 6144 floats per matrix
// Table build on the tensor cores: tensor-memory columns of a lookup CTA (the 3 stages' tables as
// 6 code tiles x 64 columns, then the codebook rows' TF32 heads and tails, 6 x 16 columns); one
// half (head or tail) of the B operand, which sits at the start of the last stage's table (that
// table is written only after every MMA has read it); the 3 mbarriers and the tensor-memory
// address behind the down input.  (Shared memory stays within the 196 KiB carveout: 4 KiB more
// there took the L1 cache from 60 to 28 KiB, and the decode step from 74.1 to 76.6 us.)
constexpr uint32_t kTmCols = 512;
constexpr uint32_t kTmA = 384;
constexpr uint32_t kBHalf = 2 * 32 * 8 * 4;
constexpr int kTcBytes = 32;
constexpr int kPrefetchRounds = 1;                 // L2 prefetch distance in row-group rounds
constexpr int kPrefetchRoundsGu = 2;               // the same for the per-phase gate/up kernel and the one-launch kernel's units

struct LutArgs {
    const uint8_t *records;
    const int32_t *slot_map; // optional expert -> record slot
    size_t stride;
    const float *codebooks;
    const int32_t *idx;
    const void *h;
    int E, k, slots;
    // gate / up: a unit is (slot, pair of consecutive 32-vector segments, matrix)
    MatGeom gu;
    size_t off_gate, off_up;
    int gu_pairs;   // segment pairs of the gate/up input, (gu.nseg + 1) / 2
    float *part_gu; // [slot][gu_pairs][2 matrices: gate, up][f]
    // down
    MatGeom dn;
    size_t off_down;
    int npair, nrb, rb_groups;
    float *part_dn; // [slot][npair][d]
    unsigned long long *stats;
    uint32_t *err;
    // optional: the slots to serve (ascending), their count on the device; null = all
    // T * k slots in order
    const int32_t *slot_list;
    const int32_t *n_list;
    // optional unit trace of the per-phase kernels: unit u of this launch writes
    // {start, tables built, end (%globaltimer ns), SM id | (ns from start to the barrier that
    // frees the tables) << 32} at trace[4 (trace_base + u)]
    unsigned long long *trace;
    int trace_cap, trace_base;
};

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Slots this launch serves.
__device__ __forceinline__ int lut_slot_count(const LutArgs &A) {
    return A.slot_list ? *A.n_list : A.slots;
}

__device__ __forceinline__ uint32_t comp(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <bool kBf16>
__device__ __forceinline__ void load_x8(const void *h, size_t elem, float *xv) {
    if constexpr (kBf16) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(h) + elem);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
            float2 f2 = __bfloat1622float2(b2);
            xv[2 * i] = f2.x;
            xv[2 * i + 1] = f2.y;
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(h) + elem);
        const float4 a = p[0], b = p[1];
        xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
        xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
    }
}

template <bool kBf16>
__device__ __forceinline__ float load_x1(const void *h, size_t elem) {
    if constexpr (kBf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(h)[elem]);
    else return reinterpret_cast<const float *>(h)[elem];
}

// Streaming load of 16 code bytes: read once, so kept out of L1.
__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void prefetch_l2_range(const uint8_t *p, size_t bytes, int lane) {
    constexpr size_t kPiece = 32768;
    for (size_t off = (size_t)lane * kPiece; off < bytes; off += 32 * kPiece) {
        const uint32_t n = (uint32_t)min(kPiece, bytes - off);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p + off), "r"(n) : "memory");
    }
}

// Slot of segment column j (0..31) within a table row of one part: the columns
// j, j + 8, j + 16, j + 24 sit side by side, so the table build stores 16 bytes at a time.
__host__ __device__ constexpr int tab_col(int j) { return 4 * (j & 7) + (j >> 3); }

// Decode a unit index into (slot, matrix, first segment, segment bases, row-group range).
// Every unit covers two consecutive 32-vector segments of one matrix (its two "parts"):
// the same rows, so both segments' lookups add into one set of row partials.
struct Unit {
    int slot, e, mat, seg0, g0, g1;
    const uint8_t *base[2]; // chunk (seg0 + p, g=0, s=0, jj=0) of each part, or null
};

// Ask L2 for row group g of both parts of a unit: 2 parts x 3 stages x 512 B = 24 lines
// of 128 B, one per lane 0..23, kept with evict_last priority until it is read.
__device__ __forceinline__ void prefetch_group(const Unit &U, int g, int lane) {
    if (lane < 24) {
        const int part = lane / 12, rest = lane % 12;
        const uint8_t *b = part ? U.base[1] : U.base[0];
        if (b) {
            const uint8_t *p = b + ((size_t)g * kStages + rest / 4) * 512 + (size_t)(rest % 4) * 128;
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
        }
    }
}

template <bool kDown>
__device__ __forceinline__ Unit decode_unit(const LutArgs &A, int u) {
    Unit U;
    if constexpr (!kDown) {
        U.slot = u / (2 * A.gu_pairs);
        if (A.slot_list) U.slot = A.slot_list[U.slot];
        const int rem = u % (2 * A.gu_pairs);
        U.seg0 = 2 * (rem >> 1);
        U.mat = rem & 1;
        U.g0 = 0;
        U.g1 = A.gu.groups;
    } else {
        const int per_slot = A.npair * A.nrb;
        U.slot = u / per_slot;
        if (A.slot_list) U.slot = A.slot_list[U.slot];
        const int rem = u % per_slot;
        U.seg0 = 2 * (rem / A.nrb);
        const int rb = rem % A.nrb;
        U.g0 = rb * A.rb_groups;
        U.g1 = min(A.dn.groups, U.g0 + A.rb_groups);
        U.mat = 2;
    }
    U.e = A.idx[U.slot];
    U.base[0] = U.base[1] = nullptr;
    const uint8_t *rec = (U.e >= 0 && U.e < A.E) ? expert_record(A.records, A.stride, A.slot_map, U.e) : nullptr;
    if (rec) {
        const MatGeom &G = kDown ? A.dn : A.gu;
        const size_t off = kDown ? A.off_down : (U.mat ? A.off_up : A.off_gate);
        for (int p = 0; p < 2; ++p)
            if (U.seg0 + p < G.nseg) U.base[p] = rec + off + (size_t)(U.seg0 + p) * G.groups * (kStages * 512);
    }
    return U;
}

// The unit's matrix codebooks (both parts: the parts are two segments of one matrix).
template <bool kDown>
__device__ __forceinline__ void unit_codebooks(const LutArgs &A, const Unit &U, const float *&p0,
                                               const float *&p1) {
    const int e = (U.e >= 0 && U.e < A.E) ? U.e : 0;
    p0 = p1 = A.codebooks + ((size_t)e * 3 + (size_t)U.mat) * kCbFloats;
}

// Table load at shared-window address a + S * 64 KiB (stage S).  volatile keeps it on
// its side of the barriers that guard the tables.
template <int S>
__device__ __forceinline__ float lds_stage(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(a), "n"(S * kTabStage));
    return v;
}

// Where the dynamic shared memory of a kernel without static shared memory starts in the
// CTA's shared window.  A lookup kernel that finds its tables there folds the table base into
// each table load's immediate offset (one instruction less per lookup); elsewhere it adds it.
constexpr uint32_t kDynSmemBase = 1024;

// Table load at shared-window address a + kDynSmemBase + S * 64 KiB: a is the prmt result
// alone (code byte and column offset), the base and stage offset the load's immediate.
template <int S>
__device__ __forceinline__ float lds_fixed(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(a), "n"(S * kTabStage + (int)kDynSmemBase));
    return v;
}

// (d0, d1) = (a0 + b0, a1 + b1) as one packed fp32 addition, each lane rounded to nearest
// like a scalar add.
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "add.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// fp32 -> TF32 by rounding the 13 dropped mantissa bits to nearest, ties away from zero:
// adding half of the kept last place to the magnitude bits and clearing the dropped bits.
// Exact for every finite input (a carry moves into the exponent as it should); the operands
// here are finite.
__device__ __forceinline__ uint32_t tf32_rna(float x) {
    return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}

// fp32 -> TF32 head plus TF32 tail (x ~ head + tail to about 2^-22 relative)
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - __uint_as_float(hi));
}


// Wait (thread 0 polls, the CTA then proceeds together) until *c >= target.  The wait
// is bounded: after limit_ns (by default about a second) it records kErrTimeout and gives up.
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void wait_counter(const unsigned *c, unsigned target, uint32_t *err,
                                             unsigned long long limit_ns = kWaitLimitNs) {
    if (threadIdx.x == 0) {
        unsigned ns = 32;
        const unsigned long long t0 = gtimer();
        while (ld_acquire(c) < target) {
            if (gtimer() - t0 > limit_ns) {
                atomicOr(err, kErrTimeout);
                break;
            }
            __nanosleep(ns);
            if (ns < 256) ns <<= 1;
        }
    }
    __syncthreads();
}

// Dynamic shared memory of the lookup kernels (every extern __shared__ array names it).
extern __shared__ __align__(16) unsigned char lut_smem[];

// Tensor-core state of a lookup CTA across its units.
struct TabTc {
    uint32_t tmem;   // tensor-memory base (kTmCols columns)
    uint32_t bar;    // shared-window address of the 3 mbarriers, one per stage
    uint32_t bbuf;   // shared-window address of the B operand (head, then tail)
    uint32_t builds; // table builds so far: the mbarriers' phase parity
};

// Every thread of the CTA, before its first unit: the mbarriers, and the tensor memory (warp 0
// allocates; one lookup CTA per SM, so the columns are free).
template <bool kRecon>
__device__ __forceinline__ void tab_tc_open(TabTc &t) {
    if constexpr (!kRecon) {
        const uint32_t off = (uint32_t)kTabBytes + (uint32_t)kXsFloats * 4;
        const uint32_t base = (uint32_t)__cvta_generic_to_shared(lut_smem);
        t.bbuf = base + (uint32_t)(kStages - 1) * kTabStage;
        t.bar = base + off;
        if (threadIdx.x == 0) {
            for (int s = 0; s < kStages; ++s) tc::mbar_init(t.bar + 8u * (uint32_t)s, 1);
            tc::mbar_init_fence();
        }
        if (threadIdx.x < 32) tc::tmem_alloc(t.bar + 8u * kStages, kTmCols);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        t.tmem = *reinterpret_cast<volatile uint32_t *>(lut_smem + off + 8 * kStages);
        t.builds = 0;
    }
}

// Every thread of the CTA, after its last unit (every table build's MMAs were waited for).
template <bool kRecon>
__device__ __forceinline__ void tab_tc_close(const TabTc &t) {
    if constexpr (!kRecon) {
        tc::fence_before_sync();
        __syncthreads();
        if (threadIdx.x < 32) {
            tc::fence_after_sync();
            tc::tmem_dealloc(t.tmem, kTmCols);
        }
    }
}

// One unit: tables (or, for the register-reconstruct form, the codebooks) for the unit's
// segments, then the stream of its rows.  `primed`: this unit's codebooks were already asked
// for by the previous unit of the CTA (else they are asked for at the start, ahead of the down
// units' input and the table build).  For a down unit, `dep` (if not null) is a completion
// counter that must reach dep_target before the gate/up partials are read.  kNT: threads of
// the CTA (a multiple of 128); kPf: L2 prefetch distance in rounds; kPartLoads: the next row
// group's codes of a part are asked for as soon as that part's lookups are issued (else at the
// top of each round -- the persistent step kernel, whose other items leave no registers for
// it); kFixed: the tables sit at kDynSmemBase (the lookups' immediate base).
template <bool kDown, bool kRecon, bool kBf16, int kNT = kThreads, int kPf = kPrefetchRounds,
          bool kPartLoads = true, bool kFixed = false>
__device__ __forceinline__ void run_unit(const LutArgs &A, const Unit &Uin, bool has_next, const Unit &Nin,
                                         bool &primed, TabTc &tcs, unsigned *dep, unsigned dep_target,
                                         unsigned long long *t_tables = nullptr, unsigned *done_prev = nullptr,
                                         unsigned *dep_used = nullptr, unsigned dep_users = 0) {
    constexpr int kNW = kNT / 32;
    static_assert(kNT % 128 == 0 && kNT <= 512, "CTA size of the lookup units");
    // the dynamic shared memory named directly, so every access compiles to a shared one
    unsigned char *smem = lut_smem;
    // local copies: the caller's structs are read once, the fields then live in registers
    const Unit U = Uin;
    Unit N = Uin;
    if (has_next) N = Nin;
    float *xs = reinterpret_cast<float *>(smem + (kRecon ? 2 * kCbFloats * 4 : kTabBytes));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const MatGeom &G = kDown ? A.dn : A.gu;
    // table column byte offset of part p: the slot of column `lane` in the permuted column
    // order of the tables
    const uint32_t colb0 = (0u << 7) | ((uint32_t)tab_col(lane) << 2);
    const uint32_t colb1 = (1u << 7) | ((uint32_t)tab_col(lane) << 2);
    const bool valid = U.base[0] != nullptr;
    // warm L2 with the first rounds of row groups this warp streams (the tail of the
    // previous unit already asked for them, except on a CTA's first unit), and with the
    // codebooks of the next unit, which its table build reads straight from global memory
#pragma unroll 1
    for (int i = 0; i < kPf; ++i) {
        const int g = U.g0 + warp + i * kNW;
        if (g < U.g1) prefetch_group(U, g, lane);
    }
    if (!kRecon && !primed && warp == 1) {
        // the CTA's first unit: its codebooks come from HBM; ask for them now, so that they
        // arrive under the down units' input and the loads of the table build hit L2
        const float *q0, *q1;
        unit_codebooks<kDown>(A, U, q0, q1);
        (void)q1;
        prefetch_l2_range(reinterpret_cast<const uint8_t *>(q0), (size_t)kCbFloats * sizeof(float), lane);
    }
    primed = !kRecon && has_next;
    if (!kRecon && has_next) {
        const float *q0, *q1;
        unit_codebooks<kDown>(A, N, q0, q1);
        constexpr int kLines = kCbFloats / 32; // 128-byte lines of one part's codebooks
        (void)q1;
        for (int i = threadIdx.x; i < kLines; i += kNT) {
            const float *q = q0 + (size_t)i * 32;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
        }
    }
    // down: a = silu(gate) * up for the 64 vectors of this unit into xs, reduced over the
    // gate/up segment pairs in a fixed order (the loads of 16 pairs in flight at a time).  It
    // reads only the slot's gate/up partials, so where nothing is waited for (the per-phase
    // kernels) it goes first, under the load of the expert index that the rest needs.
    bool input_done = false;
    auto swiglu_input = [&]() {
        __syncthreads(); // xs may still be read by the previous unit
        if (dep) wait_counter(dep, dep_target, A.err);
        for (int i = threadIdx.x; i < 2 * kSegVec * kVec; i += kNT) {
            const int r = U.seg0 * kSegVec * kVec + i; // index into f
            float a = 0.f;
            if (r < A.gu.n_out) {
                const float *pg = A.part_gu + (size_t)U.slot * A.gu_pairs * 2 * A.gu.n_out + r;
                const size_t step = (size_t)2 * A.gu.n_out;
                float zg = 0.f, zu = 0.f;
                for (int s0 = 0; s0 < A.gu_pairs; s0 += 16) {
                    float vg[16], vu[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int sg = min(s0 + q, A.gu_pairs - 1);
                        vg[q] = pg[sg * step];
                        vu[q] = pg[sg * step + A.gu.n_out];
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (s0 + q < A.gu_pairs) {
                            zg += vg[q];
                            zu += vu[q];
                        }
                }
                a = zg / (1.0f + expf(-zg)) * zu;
            }
            xs[i] = a;
        }
        __syncthreads();
        input_done = true;
    };
    if constexpr (kDown)
        if (!dep) swiglu_input();
    // Counters of a launch that runs gate/up and down units together, kept from the last warp
    // once every thread is past a barrier that follows the previous unit's partial stores (and,
    // for a down unit, its wait): done_prev counts the CTA's previous unit as finished; dep_used
    // counts this unit as a reader of dep, and the slot's last reader puts both back to zero
    // (every writer and reader of dep in this launch is then past it).
    auto counters = [&]() {
        if (threadIdx.x == kNT - 32) {
            if (done_prev) {
                __threadfence();
                atomicAdd(done_prev, 1u);
            }
            if (dep_used && atomicAdd(dep_used, 1u) == dep_users - 1) {
                *dep_used = 0u;
                *dep = 0u;
            }
        }
    };
    if (!valid) {
        // no codes to stream: the unit's rows get zero partials (the step reports the error)
        if (done_prev || dep_used) {
            if (kDown && dep && !input_done) wait_counter(dep, dep_target, A.err);
            else __syncthreads();
            counters();
        }
        if (threadIdx.x == 0) atomicOr(A.err, (U.e >= 0 && U.e < A.E) ? kErrNotResident : kErrBadExpert);
        const int r1 = min(G.n_out, U.g1 * kGroupRows);
        for (int row = U.g0 * kGroupRows + threadIdx.x; row < r1; row += kNT) {
            if constexpr (!kDown)
                A.part_gu[(((size_t)U.slot * A.gu_pairs + U.seg0 / 2) * 2 + U.mat) * G.n_out + row] = 0.f;
            else
                A.part_dn[((size_t)U.slot * A.npair + U.seg0 / 2) * G.n_out + row] = 0.f;
        }
        return;
    }
    const int t = U.slot / A.k;
    // ---- input vectors of this lane's column(s)
    float xv[2][kVec];
    if constexpr (!kDown) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int j = (U.seg0 + p) * kSegVec + lane;
            if (j < G.nv) load_x8<kBf16>(A.h, (size_t)t * A.gu.n_in + (size_t)j * kVec, xv[p]);
            else {
#pragma unroll
                for (int v = 0; v < kVec; ++v) xv[p][v] = 0.f;
            }
        }
    } else {
        if (!input_done) swiglu_input();
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
            for (int v = 0; v < kVec; ++v) xv[p][v] = xs[p * kSegVec * kVec + lane * kVec + v];
    }
    if constexpr (!kRecon) {
        // ---- tables T[s][c][part][column], one 64 KiB block per stage.  Per stage the tables
        // are the product T[c][n] = sum_v C[c][v] X[n][v] (256 codes c x 64 columns n of both
        // parts, K = 8), taken on the tensor cores by tcgen05.mma kind::tf32 into tensor memory
        // (M = 128 codes per MMA, N = 64), each operand split into a TF32 head and tail
        // (head*tail + tail*head + head*head, in that order: fp32 accuracy).  A, the codebook
        // rows, goes into tensor memory (row = lane): warp w stores the rows of its lane quarter
        // for the (stage, code tile) pairs w/4 and w/4 + 4; B, the unit's 64 input vectors, goes
        // into shared memory in the no-swizzle K-major layout, at the start of the last stage's
        // table.  Their loads are in flight across the barrier that frees the tables; the stores
        // follow it, and a second barrier precedes the MMAs.  One thread then issues the 18
        // MMAs stage by stage, each stage completing its own mbarrier,
        // and the warps copy each stage out as soon as it is complete: a 16x256b load gives the
        // registers of an mma.sync accumulator (lanes fg and fg + 8, column pairs 2 ft), so each
        // lane stores 16-byte slots of the permuted column order, conflict-free.
        static_assert(kNT == 512, "the table build maps 16 warps onto the lane quarters");
        float *tab = reinterpret_cast<float *>(smem);
        const int q = warp & 3, wg = warp >> 2;
        const int fg = lane >> 2, ft = lane & 3;
        const float *p0, *p1;
        unit_codebooks<kDown>(A, U, p0, p1);
        (void)p1;
        // A: codebook row mt * 128 + 32 q + lane of stage s for the pairs j = (s, mt) = wg, wg + 4
        float4 ca[2][2];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int j = wg + 4 * jj;
            if (j < 2 * kStages) {
                const int c = (j & 1) * 128 + q * 32 + lane;
                const float4 *r = reinterpret_cast<const float4 *>(p0 + ((size_t)(j >> 1) * kCodes + c) * kVec);
                ca[jj][0] = __ldg(r);
                ca[jj][1] = __ldg(r + 1);
            }
        }
        // B: element k = threadIdx.x % 8 of column n = threadIdx.x / 8 (part n / 32, vector n % 32)
        float xb;
        {
            const int n = threadIdx.x >> 3, k = threadIdx.x & 7;
            if constexpr (!kDown) {
                const int jg = (U.seg0 + (n >> 5)) * kSegVec + (n & 31);
                xb = jg < G.nv ? load_x1<kBf16>(A.h, (size_t)t * A.gu.n_in + (size_t)jg * kVec + k) : 0.f;
            } else {
                xb = xs[threadIdx.x];
            }
        }
        __syncthreads(); // the previous unit's lookups are done with the tables
        if (t_tables && threadIdx.x == 0) t_tables[1] = gtimer();
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int j = wg + 4 * jj;
            if (j < 2 * kStages) {
                const float v[8] = {ca[jj][0].x, ca[jj][0].y, ca[jj][0].z, ca[jj][0].w,
                                    ca[jj][1].x, ca[jj][1].y, ca[jj][1].z, ca[jj][1].w};
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) split_tf32(v[k], hi[k], lo[k]);
                const uint32_t ta = tcs.tmem + ((uint32_t)(q * 32) << 16) + kTmA + (uint32_t)j * 16;
                tc::tmem_st8(ta, hi);
                tc::tmem_st8(ta + 8, lo);
            }
        }
        {
            uint32_t hi, lo;
            split_tf32(xb, hi, lo);
            const int n = threadIdx.x >> 3, k = threadIdx.x & 7;
            const uint32_t off = (uint32_t)((n >> 3) * 256 + (k >> 2) * 128 + (n & 7) * 16 + (k & 3) * 4);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(tcs.bbuf + off), "r"(hi) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(tcs.bbuf + kBHalf + off), "r"(lo) : "memory");
        }
        tc::tmem_wait_st();
        tc::fence_proxy_async(); // B's stores, seen by the tensor core
        tc::fence_before_sync();
        __syncthreads(); // A and B staged
        tc::fence_after_sync();
        if (threadIdx.x == 0) {
            const uint32_t idesc = tc::idesc_tf32_f32(128, 2 * kSegVec);
            const uint64_t bh = tc::smem_desc(tcs.bbuf, 128, 256);
            const uint64_t bl = tc::smem_desc(tcs.bbuf + kBHalf, 128, 256);
#pragma unroll
            for (int s = 0; s < kStages; ++s) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const uint32_t d = tcs.tmem + (uint32_t)(s * 2 + mt) * 64;
                    const uint32_t a = tcs.tmem + kTmA + (uint32_t)(s * 2 + mt) * 16;
                    tc::mma_tf32_ta(d, a, bl, idesc, 0);
                    tc::mma_tf32_ta(d, a + 8, bh, idesc, 1);
                    tc::mma_tf32_ta(d, a, bh, idesc, 1);
                }
                tc::mma_commit(tcs.bar + 8u * (uint32_t)s);
            }
        }
        __syncwarp();
        // Lane (fg, ft) holds, for codes c0 + fg and c0 + fg + 8, the columns 2 ft + 8 nt (nt =
        // 0..3) -- the slots of column group 2 ft -- and 2 ft + 1 + 8 nt (group 2 ft + 1).  Lanes
        // of odd fg store group 2 ft + 1 first, so each quarter-warp's 8 lanes hit 8 different
        // bank quads in both stores.
        const int odd = fg & 1;
        const int g_first = 2 * ft + odd, g_second = 2 * ft + 1 - odd;
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            if (!tc::mbar_wait(tcs.bar + 8u * (uint32_t)s, tcs.builds & 1u)) {
                if (lane == 0) atomicOr(A.err, kErrTimeout);
                tc::mbar_wait(tcs.bar + 8u * (uint32_t)s, tcs.builds & 1u);
            }
            tc::fence_after_sync();
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                // this warp's 16 codes x 32 columns: code tile mt, half blk of its lane quarter, part mp
                const int cb = wg * 2 + i, mt = cb >> 2, blk = (cb >> 1) & 1, mp = cb & 1;
                float dd[16];
                tc::tmem_ld16x256_x4(tcs.tmem + ((uint32_t)(q * 32 + blk * 16) << 16) +
                                         (uint32_t)(s * 2 + mt) * 64 + (uint32_t)mp * kSegVec,
                                     dd);
                const int c0 = mt * 128 + q * 32 + blk * 16;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float4 ev = make_float4(dd[2 * hh], dd[4 + 2 * hh], dd[8 + 2 * hh], dd[12 + 2 * hh]);
                    float4 ov = make_float4(dd[2 * hh + 1], dd[4 + 2 * hh + 1], dd[8 + 2 * hh + 1], dd[12 + 2 * hh + 1]);
                    const int c = c0 + fg + 8 * hh;
                    float *row = tab + (((size_t)s * kCodes + c) * 2 + mp) * kSegVec;
                    *reinterpret_cast<float4 *>(row + 4 * g_first) = odd ? ov : ev;
                    *reinterpret_cast<float4 *>(row + 4 * g_second) = odd ? ev : ov;
                }
            }
        }
        ++tcs.builds;
        tc::fence_before_sync();
        __syncthreads(); // tables complete
    } else {
        __syncthreads(); // the previous unit's lookups are done with the codebook rows
        // ---- codebooks of both parts [2][3][256][8]
        const float *p0, *p1;
        unit_codebooks<kDown>(A, U, p0, p1);
        float4 *cbs = reinterpret_cast<float4 *>(smem);
        for (int i = threadIdx.x; i < 2 * kCbFloats / 4; i += kNT) {
            const float *src = (i < kCbFloats / 4) ? p0 : p1;
            const int ii = i % (kCbFloats / 4);
            cbs[i] = __ldg(reinterpret_cast<const float4 *>(src) + ii);
        }
        __syncthreads();
    }

    if (t_tables && threadIdx.x == 0) t_tables[0] = gtimer();
    // after the table barriers: the last warp's fence and atomics overlap the other warps' rows
    counters();

    // ---- stream the codes of rows [g0, g1) x this unit's segments.  L2 is asked for the row
    // group kPf rounds ahead -- past the end of the unit, for the next unit's first row groups.
    // a unit whose second segment lies past the matrix (an odd segment count) reads the first
    // segment's codes again for it: that part's tables are zero (its inputs are)
    const uint8_t *pb0 = U.base[0];
    const uint8_t *pb1 = U.base[1] ? U.base[1] : U.base[0];
    // 32-bit shared-window address of the tables: a lookup is prmt, an integer add and one
    // ld.shared with the stage offset as its immediate
    const uint32_t tab32 = (uint32_t)__cvta_generic_to_shared(smem);
    auto load_part = [&](int g, int p, uint4 (&w)[2][kStages]) {
        const uint8_t *pb = p ? pb1 : pb0;
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            const size_t co = ((size_t)g * kStages + s) * 512 + (size_t)lane * 16;
            w[p][s] = ld_stream(pb + co);
        }
    };
    auto load = [&](int g, uint4 (&w)[2][kStages]) {
        load_part(g, 0, w);
        load_part(g, 1, w);
    };
    auto ahead = [&](int g) {
        const int ga = g + kPf * kNW;
        if (ga < U.g1) prefetch_group(U, ga, lane);
        else if (has_next) {
            const int gn = N.g0 + (ga - U.g1);
            if (gn < N.g1) prefetch_group(N, gn, lane);
        }
    };
    // Row group g: lane l holds, for each code byte q of its 16-byte chunks, the partial
    // dot product of row 16 g + ((l ^ q) & 15) over its vector column.  The unit's two
    // segments add into the same 16 row partials before a single reduce-scatter over the 32
    // columns.
    auto reduce16 = [&](float (&acc)[16]) {
#pragma unroll
        for (int n = 8; n >= 2; n >>= 1)
#pragma unroll
            for (int i = 0; i < n; i += 2) {
                const float r0 = __shfl_xor_sync(0xffffffffu, acc[i + n], n);
                const float r1 = __shfl_xor_sync(0xffffffffu, acc[i + n + 1], n);
                add2(acc[i], acc[i + 1], acc[i], acc[i + 1], r0, r1);
            }
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[1], 1);
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 16);
    };
    // the lookups of part p of one row group: acc = (part 0) or += (part 1) the 16 partials.
    // Two code bytes at a time: their three stage entries are added pairwise with packed
    // additions, in the order (T0 + T1) + T2, then into the partials.  fixed: the tables sit
    // at kDynSmemBase, so a table address is the prmt result alone.
    auto lookups = [&](auto fixed, const uint4 (&cwp)[kStages], int p, float (&acc)[16]) {
        constexpr bool kFixed = decltype(fixed)::value;
        const uint32_t colb = p ? colb1 : colb0;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            const uint32_t w0 = comp(cwp[0], wd), w1 = comp(cwp[1], wd), w2 = comp(cwp[2], wd);
            if constexpr (!kRecon) {
#pragma unroll
                for (int bp = 0; bp < 2; ++bp) {
                    float t0[2], t1[2], t2[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t sel = 0x7604u | ((uint32_t)(2 * bp + h) << 4);
                        const uint32_t a0 = __byte_perm(w0, colb, sel);
                        const uint32_t a1 = __byte_perm(w1, colb, sel);
                        const uint32_t a2 = __byte_perm(w2, colb, sel);
                        if constexpr (kFixed) {
                            t0[h] = lds_fixed<0>(a0);
                            t1[h] = lds_fixed<1>(a1);
                            t2[h] = lds_fixed<2>(a2);
                        } else {
                            t0[h] = lds_stage<0>(tab32 + a0);
                            t1[h] = lds_stage<1>(tab32 + a1);
                            t2[h] = lds_stage<2>(tab32 + a2);
                        }
                    }
                    float s0, s1;
                    add2(s0, s1, t0[0], t0[1], t1[0], t1[1]);
                    add2(s0, s1, s0, s1, t2[0], t2[1]);
                    const int i = 4 * wd + 2 * bp;
                    if (p == 1) add2(acc[i], acc[i + 1], acc[i], acc[i + 1], s0, s1);
                    else {
                        acc[i] = s0;
                        acc[i + 1] = s1;
                    }
                }
            } else {
                const float *cbs = reinterpret_cast<const float *>(smem) + p * kCbFloats;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int c0 = (w0 >> (8 * b)) & 255, c1 = (w1 >> (8 * b)) & 255, c2 = (w2 >> (8 * b)) & 255;
                    const float4 *r0 = reinterpret_cast<const float4 *>(cbs + c0 * kVec);
                    const float4 *r1 = reinterpret_cast<const float4 *>(cbs + kCodes * kVec + c1 * kVec);
                    const float4 *r2 = reinterpret_cast<const float4 *>(cbs + 2 * kCodes * kVec + c2 * kVec);
                    const float4 a0 = r0[0], a1 = r0[1], b0 = r1[0], b1 = r1[1], d0 = r2[0], d1 = r2[1];
                    const float *x = xv[p];
                    float sacc = ((a0.x + b0.x) + d0.x) * x[0];
                    sacc = fmaf((a0.y + b0.y) + d0.y, x[1], sacc);
                    sacc = fmaf((a0.z + b0.z) + d0.z, x[2], sacc);
                    sacc = fmaf((a0.w + b0.w) + d0.w, x[3], sacc);
                    sacc = fmaf((a1.x + b1.x) + d1.x, x[4], sacc);
                    sacc = fmaf((a1.y + b1.y) + d1.y, x[5], sacc);
                    sacc = fmaf((a1.z + b1.z) + d1.z, x[6], sacc);
                    sacc = fmaf((a1.w + b1.w) + d1.w, x[7], sacc);
                    if (p == 1) acc[4 * wd + b] += sacc;
                    else acc[4 * wd + b] = sacc;
                }
            }
        }
    };
    // reduce-scatter of the row partials (both segments added) and store
    auto finish = [&](float (&acc)[16], int g) {
        const int row = g * kGroupRows + (lane & 15);
        reduce16(acc);
        if (lane < 16 && row < G.n_out) {
            if constexpr (!kDown)
                A.part_gu[(((size_t)U.slot * A.gu_pairs + U.seg0 / 2) * 2 + U.mat) * G.n_out + row] = acc[0];
            else
                A.part_dn[((size_t)U.slot * A.npair + U.seg0 / 2) * G.n_out + row] = acc[0];
        }
    };
    auto stream = [&](auto fixed) {
        if constexpr (!kPartLoads) {
            for (int g = U.g0 + warp; g < U.g1; g += kNW) {
                uint4 wa[2][kStages];
                load(g, wa);
                ahead(g);
                float acc[16];
                lookups(fixed, wa[0], 0, acc);
                lookups(fixed, wa[1], 1, acc);
                finish(acc, g);
            }
        } else {
            // one set of code registers: as soon as a part's lookups are issued, the next row
            // group's codes of that part are asked for into its registers, so each load has the
            // rest of the round in front of it (lines are already on their way into L2).  The
            // last round, which loads nothing, is peeled off the loop.
            uint4 wa[2][kStages];
            int g = U.g0 + warp;
            if (g < U.g1) load(g, wa);
            for (; g + kNW < U.g1; g += kNW) {
                ahead(g);
                float acc[16];
                lookups(fixed, wa[0], 0, acc);
                load_part(g + kNW, 0, wa);
                lookups(fixed, wa[1], 1, acc);
                load_part(g + kNW, 1, wa);
                finish(acc, g);
            }
            if (g < U.g1) {
                ahead(g);
                float acc[16];
                lookups(fixed, wa[0], 0, acc);
                lookups(fixed, wa[1], 1, acc);
                finish(acc, g);
            }
        }
    };
    if constexpr (!kRecon && kFixed) {
        // launched only where the tables were found at kDynSmemBase; anywhere else the
        // unit reports the mismatch and streams nothing
        if (tab32 == kDynSmemBase) stream(std::integral_constant<bool, true>{});
        else if (threadIdx.x == 0) atomicOr(A.err, kErrSmemLayout);
    } else {
        stream(std::integral_constant<bool, false>{});
    }
    // algorithmic bytes of this unit: codes of its real (row, vector) pairs,
    // and the slot's codebooks once
    if (threadIdx.x == 0 && valid && A.stats) {
        unsigned long long vecs = 0;
        for (int p = 0; p < 2; ++p) {
            const int seg = U.seg0 + p;
            if (seg < G.nseg) vecs += (unsigned long long)min(kSegVec, G.nv - seg * kSegVec);
        }
        const int rows = min(G.n_out, U.g1 * kGroupRows) - U.g0 * kGroupRows;
        atomicAdd(A.stats + kStatDemandCode, vecs * (unsigned long long)rows * kStages);
        if (U.seg0 == 0 && U.g0 == 0)
            atomicAdd(A.stats + kStatCodebook, (unsigned long long)kCbFloats * sizeof(float));
    }
}

// Bytes of dynamic shared memory of a unit.
template <bool kRecon>
constexpr size_t unit_smem() {
    return (kRecon ? 2 * kCbFloats * 4 : kTabBytes) + kXsFloats * 4 + (kRecon ? 0 : kTcBytes);
}

} // namespace lut
} // namespace wm
