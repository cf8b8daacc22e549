// Expert matrices applied straight from their RVQ codes, one (token, expert)
// slot at a time: the decode path.
//
// Method (page "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s", section
// "Quantification et exactitude"): the weights are stored as 3 residual stages
// of 256-entry codebooks over 8-weight vectors, and the product is taken
// without rebuilding the matrix -- a table of partial dot products
// T[s][j][c] = <C_s[c], x_j> is built, then each row costs 3 lookups and 2
// additions per vector.
//
// GB300 mapping.  A CTA (512 threads, one per SM, persistent) owns a "unit":
// one slot, one matrix and two consecutive 32-vector segments of its input (for
// down also a block of rows).  It builds the unit's tables in shared memory --
// T[s][c][part][lane], 3 x 64 KiB, so that lane l always reads bank l whatever
// the code -- then streams all rows' codes of those segments with 128-bit
// loads.  Each lane owns one vector column of each segment and 16 rows per
// 16-byte chunk; the chunk's bytes are pre-permuted (row (lane ^ q) & 15 at byte
// q) so the cross-lane reduction of 32 row partials is a select-free butterfly.
// One prmt turns a code byte plus the lane's column offset into the table
// address (the tables' base and the stage in the load's immediate), so a lookup
// costs a prmt, an ld.shared and half of a packed fp32 addition.
// Partials of each segment go to a scratch buffer; a down unit reduces the
// gate/up partials of its slot in a fixed order, applies SwiGLU and builds its
// own tables; a last kernel combines the k expert outputs with their gates.  A
// handle's forward runs the gate/up and the down units in one launch (each down
// unit waits for its slot's gate/up units); the per-phase kernels, one launch
// per phase, serve the listed slots of batched calls, the reconstruct form and
// the no-allocation entry point.  Every sum has a fixed order: results are
// bit-reproducible, and the same in either form.
//
// The K2_RECONSTRUCT variant instead stages the codebooks in shared memory and
// rebuilds each 8-weight vector in registers (3 codebook rows summed) before an
// 8-term dot product.
#include "lut_dev.cuh"

namespace wm {

using namespace lut;

namespace {

// Per-unit trace entry {start, tables ready, end, SM | table-barrier wait << 32}.
__device__ __forceinline__ void trace_unit(const LutArgs &A, int item, unsigned long long t0,
                                           const unsigned long long (&t_tab)[2]) {
    if (A.trace && threadIdx.x == 0 && A.trace_base + item < A.trace_cap) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        unsigned long long *e = A.trace + 4 * (size_t)(A.trace_base + item);
        e[0] = t0;
        e[1] = t_tab[0];
        e[2] = gtimer();
        e[3] = smid | ((t_tab[1] > t0 ? (t_tab[1] - t0) : 0ull) << 32);
    }
}

template <bool kDown, bool kRecon, bool kBf16, int kNT, int kPf, bool kFixed>
__global__ void __launch_bounds__(kNT, 1) lut_kernel(const LutArgs A) {
    const int n_slots = lut_slot_count(A);
    const int units = kDown ? n_slots * A.npair * A.nrb : n_slots * 2 * A.gu_pairs;
    bool primed = false;
    TabTc tcs;
    tab_tc_open<kRecon>(tcs);
    Unit N;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const Unit U = decode_unit<kDown>(A, u);
        const bool has_next = u + (int)gridDim.x < units;
        if (has_next) N = decode_unit<kDown>(A, u + gridDim.x);
        unsigned long long t0 = 0, t_tab[2] = {0, 0};
        if (A.trace && threadIdx.x == 0) t0 = gtimer();
        run_unit<kDown, kRecon, kBf16, kNT, kPf, true, kFixed>(A, U, has_next, N, primed, tcs, nullptr, 0,
                                                               A.trace ? t_tab : nullptr);
        trace_unit(A, u, t0, t_tab);
    }
    tab_tc_close<kRecon>(tcs);
}

// The gate/up and the down units of one call in one launch, so that a CTA starts its down
// unit as soon as its own gate/up units and those of the down unit's slot are done, with no
// kernel boundary between the two phases.  CTA b runs gate/up units b, b + G, ... and then
// down units G - 1 - b, 2 G - 1 - b, ...: the CTAs with one gate/up unit fewer take the
// first slots' down units, whose gate/up units finish first.  A down unit waits (bounded) on
// its slot's count of finished gate/up units, so every CTA must be resident at once: the
// launch is cooperative.  sync: [4 + slot] gate/up units of the slot finished, [4 + slots +
// slot] its down units past that wait; zero at rest, and the slot's last down unit puts both
// back.  A finished gate/up unit is counted inside the CTA's next unit, once its tables are
// built, so that the fence of the count runs beside that unit's rows (the CTA's last gate/up
// unit is counted before its first down unit).  Same unit arithmetic as the per-phase kernels:
// the results are bit-identical to theirs.
// The lookahead's share of lookahead CTA k of n_la (inside the one-launch expert kernel): the
// next layer's top-P experts, selected from its selection keys by rank (the number of keys that
// come first in the router's own order: larger key, or equal key and smaller index) -- each
// lookahead CTA takes the same selection by itself, so none waits for another -- then CTA k's
// share of the predicted experts' pieces asked of L2.  CTA 0 also stores the prediction.
__device__ __noinline__ void lookahead_item(const LutAhead LA, int k, int n_la) {
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(lut_smem); // [E]
    int *sel = reinterpret_cast<int *>(lut_smem + 8 * kThreads);                 // [P]
    __syncthreads(); // the CTA's last unit is done with its shared memory
    for (int i = threadIdx.x; i < LA.E; i += kThreads) keys[i] = LA.keys[i];
    __syncthreads();
    for (int i = threadIdx.x; i < LA.E; i += kThreads) {
        const unsigned long long ki = keys[i];
        int rank = 0;
        for (int j = 0; j < LA.E; ++j) {
            const unsigned long long kj = keys[j];
            rank += (kj > ki || (kj == ki && j < i)) ? 1 : 0;
        }
        if (rank < LA.P) sel[rank] = i;
    }
    __syncthreads();
    if (k == 0) {
        if ((int)threadIdx.x < LA.P) LA.pred_idx[threadIdx.x] = sel[threadIdx.x];
        if (threadIdx.x == 0) {
            *LA.pred_count = LA.P;
            if (LA.stats) {
                atomicAdd(LA.stats + kStatPrefetchBytes, (unsigned long long)LA.P * lookahead_bytes(LA.nseg, LA.groups));
                atomicAdd(LA.stats + kStatPrefetchExperts, (unsigned long long)LA.P);
            }
        }
    }
    const int per = lookahead_pieces(LA.nseg);
    for (int j = k + n_la * (int)threadIdx.x; j < LA.P * per; j += n_la * kThreads)
        lookahead_piece(LA.records, LA.stride, LA.off_gate, LA.off_up, LA.nseg, LA.groups, LA.codebooks, sel[j / per],
                        j % per);
}

// kAhead: the launch carries the lookahead, in its own instance and out of line (its code inside
// every instance cost 1.5 us of the one-layer step; inlined into its own instance, 0.2 us per
// layer of the stack)
template <bool kBf16, bool kFixed, bool kAhead>
__global__ void __launch_bounds__(kThreads, 1) lut_experts_kernel(const LutArgs A, unsigned *sync, const LutAhead LA) {
    const int n_gu = A.slots * 2 * A.gu_pairs;
    const int n_dn = A.slots * A.npair * A.nrb;
    const int G = gridDim.x, b = blockIdx.x;
    const int mine_gu = b < n_gu ? (n_gu - 1 - b) / G + 1 : 0;
    const int d0 = G - 1 - b;
    const int mine_dn = d0 < n_dn ? (n_dn - 1 - d0) / G + 1 : 0;
    bool primed = false;
    TabTc tcs;
    tab_tc_open<false>(tcs);
    // slot counter of the CTA's last finished gate/up unit, bumped inside the next unit (once
    // its tables are built), or before the first down unit
    int pending = -1;
    for (int i = 0; i < mine_gu; ++i) {
        const int u = b + i * G;
        // the next unit: the CTA's next gate/up unit, else its first down unit
        const bool has_next = i + 1 < mine_gu || mine_dn > 0;
        Unit N;
        if (i + 1 < mine_gu) N = decode_unit<false>(A, u + G);
        else if (mine_dn > 0) N = decode_unit<true>(A, d0);
        unsigned long long t0 = 0, t_tab[2] = {0, 0};
        if (A.trace && threadIdx.x == 0) t0 = gtimer();
        const Unit U = decode_unit<false>(A, u);
        run_unit<false, false, kBf16, kThreads, kPrefetchRoundsGu, true, kFixed>(
            A, U, has_next, N, primed, tcs, nullptr, 0, A.trace ? t_tab : nullptr,
            pending >= 0 ? sync + 4 + pending : nullptr);
        trace_unit(A, u, t0, t_tab);
        pending = U.slot;
    }
    if (pending >= 0) {
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(sync + 4 + pending, 1u);
        }
    }
    // the lookahead: the CTAs without a down unit (or, if every CTA has one, CTA 0 at its end)
    const int n_la = n_dn < G ? G - n_dn : 1;
    if constexpr (kAhead)
        if (n_dn < G && mine_dn == 0) lookahead_item(LA, b, n_la);
    for (int i = 0; i < mine_dn; ++i) {
        const int u = d0 + i * G;
        const bool has_next = i + 1 < mine_dn;
        Unit N;
        if (has_next) N = decode_unit<true>(A, u + G);
        unsigned long long t0 = 0, t_tab[2] = {0, 0};
        if (A.trace && threadIdx.x == 0) t0 = gtimer();
        const Unit U = decode_unit<true>(A, u);
        // L2 asked for two rounds ahead here (one in the per-phase down kernel): in this launch
        // the down units stream beside fewer others (one box: step 72.97 -> 72.49 us; three: 72.5)
        run_unit<true, false, kBf16, kThreads, kPrefetchRoundsGu, true, kFixed>(
            A, U, has_next, N, primed, tcs, sync + 4 + U.slot, (unsigned)(2 * A.gu_pairs), A.trace ? t_tab : nullptr,
            nullptr, sync + 4 + A.slots + U.slot, (unsigned)(A.npair * A.nrb));
        trace_unit(A, n_gu + u, t0, t_tab);
    }
    if constexpr (kAhead)
        if (n_dn >= G && b == 0) lookahead_item(LA, 0, 1);
    tab_tc_close<false>(tcs);
}

// out[t] (mode 0: =, 1: +=, 2: = h +) sum_i gate[t][i] * sum_pair part_dn[t*k+i][pair],
// slots in rank order and pairs in order.  A CTA takes 32 rows of one token with one warp per
// slot: lane l of warp i sums slot i's pairs of row l (every load of the launch in flight at
// once, one round trip), and warp 0 adds the slots in rank order.  NP = number of pairs (0:
// any, read in a loop).  one_part: slots whose single partial is their whole output (the
// tensor-core slots of a batched call).
template <int NP>
__global__ void __launch_bounds__(32 * kMaxTopK) combine_kernel(const float *__restrict__ part_dn,
                                                                const int32_t *__restrict__ idx,
                                                                const float *__restrict__ gate,
                                                                const float *__restrict__ h,
                                                                float *__restrict__ out, int d, int k, int E,
                                                                int npair_rt, int mode,
                                                                unsigned long long *stats,
                                                                unsigned long long slots,
                                                                const uint8_t *__restrict__ one_part) {
    __shared__ float sv[kMaxTopK][32];
    __shared__ float gs[kMaxTopK];
    __shared__ int oks[kMaxTopK];
    const int t = blockIdx.y;
    const int i = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 32 + lane;
    if (stats && blockIdx.x == 0 && t == 0 && threadIdx.x == 0) atomicAdd(stats + kStatForwardSlots, slots);
    const int npair = NP ? NP : npair_rt;
    const size_t si = (size_t)t * k + i;
    if (r < d) {
        const float *p = part_dn + si * npair * d + r;
        float s = 0.f;
        if constexpr (NP > 0) {
            float pv[NP];
#pragma unroll
            for (int q = 0; q < NP; ++q) pv[q] = p[(size_t)q * d];
#pragma unroll
            for (int q = 0; q < NP; ++q) s += pv[q];
            if (one_part && one_part[si]) s = pv[0];
        } else {
            const int nq = (one_part && one_part[si]) ? 1 : npair;
            for (int q = 0; q < nq; ++q) s += p[(size_t)q * d];
        }
        sv[i][lane] = s;
    }
    if (lane == 0) {
        const int e = idx[si];
        oks[i] = e >= 0 && e < E;
        gs[i] = gate[si];
    }
    __syncthreads();
    if (i != 0 || r >= d) return;
    float y = 0.f;
    for (int j = 0; j < k; ++j)
        if (oks[j]) y = fmaf(gs[j], sv[j][lane], y);
    const size_t o = (size_t)t * d + r;
    if (mode == 0) out[o] = y;
    else if (mode == 1) out[o] = out[o] + y;
    else out[o] = h[o] + y;
}

// Where a kernel without static shared memory finds its dynamic shared memory: written by a
// one-thread probe, read once per device.
__device__ unsigned g_dyn_smem_base;

__global__ void smem_base_probe_kernel() {
    if (threadIdx.x == 0) g_dyn_smem_base = (unsigned)__cvta_generic_to_shared(lut_smem);
}

// 0: not probed yet, 1: the tables sit at kDynSmemBase, 2: elsewhere.
std::atomic<int> g_tables_fixed[kMaxDevices];

// Whether the lookup kernels of the current device find their tables at kDynSmemBase (then
// they take the table base as a load immediate).  Probed on stream s the first time it is
// asked outside a stream capture; a captured call before that takes the general kernels.
bool tables_at_fixed_base(cudaStream_t s) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    const int known = g_tables_fixed[dev].load(std::memory_order_acquire);
    if (known) return known == 1;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return false;
    const int smem = (int)unit_smem<false>();
    static SmemAttr attr;
    if (ensure_smem(attr, (const void *)smem_base_probe_kernel, smem) != cudaSuccess) return false;
    smem_base_probe_kernel<<<1, 32, smem, s>>>();
    unsigned base = ~0u;
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&base, g_dyn_smem_base, sizeof base, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return false;
    g_tables_fixed[dev].store(base == kDynSmemBase ? 1 : 2, std::memory_order_release);
    return base == kDynSmemBase;
}

template <bool kDown, bool kRecon, bool kBf16, int kNT, int kPf, bool kFixed>
cudaError_t launch_v(const LutArgs &A, int units, int num_sms, cudaStream_t s) {
    const size_t smem = unit_smem<kRecon>();
    static SmemAttr attr;
    cudaError_t e =
        ensure_smem(attr, (const void *)lut_kernel<kDown, kRecon, kBf16, kNT, kPf, kFixed>, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = units < num_sms ? units : num_sms;
    lut_kernel<kDown, kRecon, kBf16, kNT, kPf, kFixed><<<grid, kNT, smem, s>>>(A);
    return cudaGetLastError();
}

// The per-phase lookup kernels: 512 threads; the next round's codes of a part are loaded
// as soon as that part's lookups are issued, and L2 is asked for the rounds ahead (measured
// on GB300 at the decode shape, same box, interleaved runs: gate/up 42.9 us with L2 two
// rounds ahead against 44.3 with one; down 24.6 us with one against 26.6 with two; earlier,
// before the lookups took fewer instructions, one round was best for both; 384 threads with
// a second register set for the codes were slower).
template <bool kDown, bool kRecon, bool kBf16>
cudaError_t launch_one(const LutArgs &A, int units, int num_sms, cudaStream_t s) {
    constexpr int kPf = kDown ? kPrefetchRounds : kPrefetchRoundsGu;
    if constexpr (!kRecon)
        if (tables_at_fixed_base(s))
            return launch_v<kDown, false, kBf16, kThreads, kPf, true>(A, units, num_sms, s);
    return launch_v<kDown, kRecon, kBf16, kThreads, kPf, false>(A, units, num_sms, s);
}

template <bool kDown>
cudaError_t launch_var(const LutArgs &A, int units, bool recon, bool bf16, int num_sms, cudaStream_t s) {
    if (recon) return bf16 ? launch_one<kDown, true, true>(A, units, num_sms, s)
                           : launch_one<kDown, true, false>(A, units, num_sms, s);
    return bf16 ? launch_one<kDown, false, true>(A, units, num_sms, s)
                : launch_one<kDown, false, false>(A, units, num_sms, s);
}

// Whether the current device takes cooperative launches (asked once per device).
bool coop_launch_ok() {
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
    return c == 1;
}

template <bool kBf16, bool kFixed, bool kAhead>
cudaError_t launch_experts_v(const LutArgs &A, unsigned *sync, const LutAhead &LA, int grid, cudaStream_t s) {
    const size_t smem = unit_smem<false>();
    static SmemAttr attr;
    cudaError_t e = ensure_smem(attr, (const void *)lut_experts_kernel<kBf16, kFixed, kAhead>, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, lut_experts_kernel<kBf16, kFixed, kAhead>, A, sync, LA);
}

// The gate/up and down units in one cooperative launch of at most one CTA per SM.
cudaError_t launch_experts(const LutArgs &A, unsigned *sync, const LutAhead &LA, bool bf16, int num_sms,
                           cudaStream_t s) {
    const int n_gu = A.slots * 2 * A.gu_pairs, n_dn = A.slots * A.npair * A.nrb;
    const int units = n_gu > n_dn ? n_gu : n_dn;
    const int grid = units < num_sms ? units : num_sms;
    const bool ahead = LA.keys != nullptr;
    if (tables_at_fixed_base(s)) {
        if (ahead)
            return bf16 ? launch_experts_v<true, true, true>(A, sync, LA, grid, s)
                        : launch_experts_v<false, true, true>(A, sync, LA, grid, s);
        return bf16 ? launch_experts_v<true, true, false>(A, sync, LA, grid, s)
                    : launch_experts_v<false, true, false>(A, sync, LA, grid, s);
    }
    if (ahead)
        return bf16 ? launch_experts_v<true, false, true>(A, sync, LA, grid, s)
                    : launch_experts_v<false, false, true>(A, sync, LA, grid, s);
    return bf16 ? launch_experts_v<true, false, false>(A, sync, LA, grid, s)
                : launch_experts_v<false, false, false>(A, sync, LA, grid, s);
}

} // namespace

// Row blocks of the down matrix per (slot, segment pair): enough units to fill
// the SMs, but at least 64 row groups per unit so the table build stays small
// next to the rows it serves.
int down_row_blocks(int slots, int npair, int groups, int num_sms) {
    const int base = slots * npair;
    int nrb = (num_sms + base / 2) / base;
    const int max_rb = groups / 64 > 1 ? groups / 64 : 1;
    if (nrb > max_rb) nrb = max_rb;
    if (nrb < 1) nrb = 1;
    return nrb;
}

LutArgs make_lut_args(const LayerView &L, const Workspace &W, const void *h, int T,
                      const int32_t *idx, int num_sms) {
    LutArgs A;
    A.records = L.records;
    A.slot_map = L.slot_map;
    A.stride = L.stride;
    A.codebooks = L.codebooks;
    A.idx = idx;
    A.h = h;
    A.E = L.E;
    A.k = L.k;
    A.slots = T * L.k;
    A.gu = L.gu;
    A.off_gate = L.sec_off[0];
    A.off_up = L.sec_off[1];
    A.gu_pairs = (L.gu.nseg + 1) / 2;
    A.part_gu = W.part_gu;
    A.dn = L.dn;
    A.off_down = L.sec_off[2];
    A.npair = (L.dn.nseg + 1) / 2;
    A.nrb = down_row_blocks(A.slots, A.npair, L.dn.groups, num_sms);
    A.rb_groups = (L.dn.groups + A.nrb - 1) / A.nrb;
    A.part_dn = W.part_dn;
    A.stats = W.stats;
    A.err = W.err;
    A.slot_list = nullptr;
    A.n_list = nullptr;
    A.trace = nullptr;
    A.trace_cap = 0;
    A.trace_base = 0;
    return A;
}

cudaError_t launch_lut_phase(const LutArgs &A, bool down, bool reconstruct, bool bf16, int num_sms,
                             cudaStream_t s) {
    if (!down) return launch_var<false>(A, A.slots * 2 * A.gu_pairs, reconstruct, bf16, num_sms, s);
    return launch_var<true>(A, A.slots * A.npair * A.nrb, reconstruct, bf16, num_sms, s);
}

cudaError_t launch_lut_listed(const LayerView &L, const Workspace &W, const void *h, int T,
                              const int32_t *idx, const int32_t *slot_list, const int32_t *n_list,
                              bool down, bool reconstruct, int num_sms, cudaStream_t s) {
    LutArgs A = make_lut_args(L, W, h, T, idx, num_sms);
    A.slot_list = slot_list;
    A.n_list = n_list;
    return launch_lut_phase(A, down, reconstruct, L.act_bf16 != 0, num_sms, s);
}

cudaError_t launch_combine(const LayerView &L, const Workspace &W, const void *h, int T,
                           const int32_t *idx, const float *gate, float *out, int mode,
                           const uint8_t *one_part, int nparts, cudaStream_t s) {
    const unsigned long long slots = (unsigned long long)T * L.k;
    dim3 grid((L.d + 31) / 32, T);
    const float *h32 = reinterpret_cast<const float *>(h);
    switch (nparts) {
#define WM_COMBINE(NP)                                                                               \
    combine_kernel<NP><<<grid, 32 * L.k, 0, s>>>(W.part_dn, idx, gate, h32, out, L.d, L.k, L.E, nparts, \
                                                        mode, W.stats, slots, one_part)
    case 1: WM_COMBINE(1); break;
    case 2: WM_COMBINE(2); break;
    case 3: WM_COMBINE(3); break;
    case 4: WM_COMBINE(4); break;
    case 5: WM_COMBINE(5); break;
    case 6: WM_COMBINE(6); break;
    case 7: WM_COMBINE(7); break;
    case 8: WM_COMBINE(8); break;
    default: WM_COMBINE(0); break;
#undef WM_COMBINE
    }
    return cudaGetLastError();
}

cudaError_t launch_lut_forward(const LayerView &L, const Workspace &W, const void *h, int T,
                               const int32_t *idx, const float *gate, float *out, int mode,
                               bool reconstruct, int num_sms, cudaStream_t s, Timing *tm,
                               unsigned long long *trace, int trace_cap, const LutAhead *ahead) {
    LutArgs A = make_lut_args(L, W, h, T, idx, num_sms);
    A.trace = trace;
    A.trace_cap = trace ? trace_cap : 0;
    const bool bf16 = L.act_bf16 != 0;
    if (tm) cudaEventRecord(tm->ev[0], s);
    if (!reconstruct && W.sync && coop_launch_ok()) {
        // gate/up and down units in one launch, then the combine
        A.trace_base = 0;
        LutAhead LA{};
        if (ahead && ahead->keys && T == 1 && ahead->E <= kThreads && ahead->P >= 1 && ahead->P <= kMaxTopK)
            LA = *ahead;
        cudaError_t e = launch_experts(A, W.sync, LA, bf16, num_sms, s);
        if (e != cudaSuccess) return e;
        if (tm) cudaEventRecord(tm->ev[1], s);
        e = launch_combine(L, W, h, T, idx, gate, out, mode, nullptr, down_parts(L), s);
        if (e != cudaSuccess) return e;
        if (tm) {
            cudaEventRecord(tm->ev[2], s);
            tm->n = 3;
        }
        return cudaSuccess;
    }
    cudaError_t e = launch_lut_phase(A, false, reconstruct, bf16, num_sms, s);
    if (e != cudaSuccess) return e;
    if (tm) cudaEventRecord(tm->ev[1], s);
    A.trace_base = A.slots * 2 * A.gu_pairs; // down units follow the gate/up units
    e = launch_lut_phase(A, true, reconstruct, bf16, num_sms, s);
    if (e != cudaSuccess) return e;
    if (tm) cudaEventRecord(tm->ev[2], s);
    e = launch_combine(L, W, h, T, idx, gate, out, mode, nullptr, down_parts(L), s);
    if (e != cudaSuccess) return e;
    if (tm) {
        cudaEventRecord(tm->ev[3], s);
        tm->n = 4;
    }
    return cudaSuccess;
}

} // namespace wm
