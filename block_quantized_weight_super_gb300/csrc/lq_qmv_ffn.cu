// lq_qmv_ffn.cu -- the whole batch-1 FFN in one launch: gate/up pairs with
// the gated activation (phase 0), then the down projection of the h that
// phase 0 wrote (phase 1).  larql "Architecture -> Metal shader map", Gemma 3
// table: q4k_ffn_gate_up + geglu followed by the Q6_K down projection; the
// pages run these as separate dispatches.
//
// Every CTA takes its tiles of phase 0 (tiles [0, T0), dealt round robin over
// the grid), then its tiles of phase 1.  The producer warp streams the tiles
// of both phases through one ring of stages without a break, so the first
// down tiles are in shared memory while the last gate/up tiles are computed;
// separate launches pay a ramp and a drain for each matrix instead.  The
// producer sums the partials of the phase-0 tiles but the last two, which the
// consumer warps share; once the producer has signalled that its share of h
// is written, consumer thread 0 arrives on a grid barrier and waits for every
// CTA, then bulk-copies h into shared memory as x of phase 1.  The work
// items, the reductions and so every result are those of the separate
// gate/up and down launches, bit for bit.  On GB300 at the Gemma-3-4B FFN
// this is not faster than the two launches: the barrier and the distribution
// of h to every CTA cost what the second launch did.
//
// Grid barrier: one device word whose low 31 bits are zero between calls
// (zero before its first use).  CTA 0 adds 2^31 - (grid - 1) and every other
// CTA adds 1: whatever the order, the low bits stay below 2^31 until the last
// arrival, which carries into the top bit and leaves the low bits zero again.
// So the top bit flips exactly when all CTAs have arrived, and nothing is
// reset.  Every CTA arrives exactly once, also when it gave up.
// All CTAs of the grid must be resident at once: the host sizes the grid by
// the occupancy, and the CTAs of the preceding kernel leave as these start.
// Waits are bounded like every other wait (STATUS_TIMEOUT).
#include "lq_qmv_impl.cuh"

namespace lq {
namespace {

__device__ __forceinline__ int phase_tiles(int first, int step, int ntile) {
    return first < ntile ? (ntile - 1 - first) / step + 1 : 0;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded) until the barrier word's top bit differs from that of `old`.
__device__ __forceinline__ bool grid_wait(const unsigned* bar, uint32_t old, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (((ld_acquire_gpu(bar) ^ old) & 0x80000000u) == 0) {
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

struct FfnState {
    int s, slot_n;
    uint32_t fphase;
    uint32_t xn;            // bulk stagings of x so far (parity of the next)
    bool aborted;
};

// The consumers' share of one phase: stage x, then the work items of each of
// the phase's tiles of this CTA (tiles first, first + step, ...).
template <int FMT, int R, bool COHERENT>
__device__ __forceinline__ void ffn_consume(const QmvParams& P, const GroupConsts& K, const Smem& sm,
                                            const QGeo& Gm, const Seg& S, int ntl, int NCT, int red_tile,
                                            FfnState& st) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int S_ = P.nstages, NRED = S_ + 1;
    const int U = Gm.U, UP = Gm.UP, half = Gm.RT / 2;
    const int rb = (int)qrow_bytes(FMT, Gm.cols);
    const int G_first = tid % U, row_first = (tid / U) * R;
    consumer_sync(NCT);                  // every consumer is done with the previous x (and,
                                         // in phase 1, warp 0 has seen the grid barrier)
    // x of phase 0 (from the preceding kernel) by loads, which start before the
    // weight tiles already queued on the bulk-copy engine; h (phase 1) by bulk
    // copies, issued once the grid barrier has passed
    bool ok = true;
    if (COHERENT) {
        ok = stage_x_bulk<FMT, 1>(Gm, S, sm.xs, sm.sxs, sm.xfull, st.xn & 1u, P.timeout_ns, tid, NCT, true);
        ++st.xn;
    } else {
        stage_x<FMT, 1>(Gm, S, sm.xs, sm.sxs, tid, NCT);
    }
    if (!ok && !st.aborted) {
        st.aborted = true;
        if (lane == 0) {
            record_status(P.status, STATUS_TIMEOUT);
            atomicExch(sm.abort_flag, 1);
        }
    }
    const int dG = NCT % U, dRow = (NCT / U) * R;
    for (int k = 0; k < ntl; ++k) {
        const int s = st.s;
        if (!st.aborted) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(&sm.full[s], (st.fphase >> s) & 1u, P.timeout_ns);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok || warp_aborted(sm.abort_flag, lane)) {
                st.aborted = true;
                if (lane == 0 && !ok) {
                    record_status(P.status, STATUS_TIMEOUT);
                    atomicExch(sm.abort_flag, 1);
                }
            }
        }
        st.fphase ^= 1u << s;
        const uint8_t* stg = sm.stages + (size_t)s * P.stage_bytes;
        float* red = sm.red + (size_t)st.slot_n * red_tile;
        if (!st.aborted) {
            int G = G_first, row0 = row_first;
            for (int q = 0; q < Gm.ipt; ++q) {
                const uint8_t* rp[R];
#pragma unroll
                for (int r = 0; r < R; ++r) rp[r] = stg + (row0 + r) * rb;
                float part[R][1];
                const Q4Sel sel = q4_sel(G & 3);
                run_item<FMT, 1, R>(rp, G, sm.xs, sm.sxs, U, sel, K, part);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int rho = row0 + r;
                    const int slot = S.mode == MODE_PAIR_INTERLEAVED ? (rho & 1) * half + (rho >> 1) : rho;
                    red[slot * UP + G] = part[r][0];
                }
                G += dG;
                row0 += dRow;
                if (G >= U) {
                    G -= U;
                    row0 += R;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
        if (++st.s == S_) st.s = 0;
        if (++st.slot_n == NRED) st.slot_n = 0;
    }
}

template <int F0, int R0, int F1, int R1>
__device__ void qmv_ffn_cta(const QmvParams& P, const GroupConsts& K, const Smem& sm, uint64_t* gready) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NC = (blockDim.x >> 5) - 1;
    const int NCT = NC * 32;
    const int S_ = P.nstages, NRED = S_ + 1;
    const int red_tile = P.red_tile;
    const int bid = blockIdx.x, grid = gridDim.x;
    const int T0 = P.tile_split;
    const int N0 = phase_tiles(bid, grid, T0), N1 = phase_tiles(bid, grid, P.ntiles - T0);
    const int NT = N0 + N1;
    // Who sums which tile's partials: the consumer warps share the last two
    // tiles of each phase ([P0, N0) and [P1, NT)), the producer the others.
    const int P0 = max(0, N0 - 2), P1 = max(N0, NT - 2);
    auto by_producer = [&](int m) { return m < P0 || (m >= N0 && m < P1); };
    // tile of this CTA's n-th position: phase 0 first
    auto tile_of = [&](int n) { return n < N0 ? bid + n * grid : T0 + bid + (n - N0) * grid; };
    // the consumers released tile m (its partials are complete): the m / S-th
    // completion of its stage's empty barrier, waited for before tile m + S
    // is issued, so the barrier is never a full two phases ahead
    auto wait_empty = [&](int m) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(&sm.empty[m % S_], (uint32_t)(m / S_) & 1u, P.timeout_ns);
        return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
    };

    if (warp == NC) {
        // ------------------------------------------------ producer warp
        const uint64_t policy = policy_evict_first();
        int last_use[8];
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) last_use[s2] = -1;
        bool ok = true, ready = false;
        int ntiles = 0;
        auto reduce = [&](int m) {
            const bool ph = m >= N0;
            __syncwarp();
            reduce_tile<1>(P.geo[ph ? 1 : 0], sm.segs[ph ? 1 : 0], tile_of(m),
                           sm.red + (size_t)(m % NRED) * red_tile, lane, 0, 1);
        };
        // tell the consumers once every phase-0 tile of the producer's share is
        // summed (its h written and fenced); they arrive on the grid barrier
        auto signal_ready = [&](int done) {
            if (ready || done < P0) return;
            __threadfence();
            __syncwarp();
            if (lane == 0) mbar_arrive(gready);
            ready = true;
        };
        for (int n = 0, s = 0; n < NT; ++n) {
            if (n == S_) pdl_wait();      // stages full: the rest waits for the preceding kernel
            if (warp_aborted(sm.abort_flag, lane)) break;
            if (n >= S_ && !(ok = wait_empty(n - S_))) break;
            const int ph = n >= N0 ? 1 : 0;
            const QTile g = qtile(P.geo[ph], sm.segs[ph], tile_of(n));
            uint8_t* dst = sm.stages + (size_t)s * P.stage_bytes;
            if (g.tma) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.full[s], g.bytes1);
                    bulk_g2s_stream(dst, g.src1, g.bytes1, &sm.full[s], policy);
                }
                last_use[s] = n / S_;
            } else {
                warp_copy(dst, g.src1, g.bytes1, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.full[s]);
            }
            if (n >= S_ && by_producer(n - S_)) reduce(n - S_);
            if (n >= S_) signal_ready(n - S_ + 1);
            if (++s == S_) s = 0;
            ntiles = n + 1;
        }
        if (ntiles <= S_) pdl_wait();     // (the loop waited iff it reached tile S)
        // the producer's tiles among the last S issued
        for (int m = max(0, ntiles - S_); ok && m < ntiles; ++m) {
            signal_ready(m);
            if (!by_producer(m)) continue;
            if (warp_aborted(sm.abort_flag, lane)) break;
            if (!(ok = wait_empty(m))) break;
            reduce(m);
        }
        if (!ok && lane == 0) {
            record_status(P.status, STATUS_TIMEOUT);
            atomicExch(sm.abort_flag, 1);
        }
        signal_ready(1 << 30);            // also when it gave up: the consumers never wait in vain
        if (lane == 0) {
            for (int s2 = 0; s2 < S_; ++s2)
                if (last_use[s2] >= 0)
                    mbar_wait_bounded(&sm.full[s2], (uint32_t)last_use[s2] & 1u, P.timeout_ns);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    pdl_wait();                           // x comes from the preceding kernel
    FfnState st{0, 0, 0u, 0u, false};
    // the consumers' share of the reductions: tiles [m0, m1) of phase ph
    auto reduce_last = [&](int m0, int m1, int ph) {
        for (int m = m0; m < m1 && !st.aborted; ++m) {
            const int k = m - (m1 - 2);
            if (!wait_empty(m)) {
                st.aborted = true;
                if (lane == 0) {
                    record_status(P.status, STATUS_TIMEOUT);
                    atomicExch(sm.abort_flag, 1);
                }
                break;
            }
            reduce_tile<1>(P.geo[ph], sm.segs[ph], tile_of(m), sm.red + (size_t)(m % NRED) * red_tile, lane,
                           k ? NC - 1 - warp : warp, NC);
        }
    };
    if (N0 > 0) {
        ffn_consume<F0, R0, false>(P, K, sm, P.geo[0], sm.segs[0], N0, NCT, red_tile, st);
        reduce_last(P0, N0, 0);
    }
    // This CTA's h is written (the consumers' share fenced here, the
    // producer's before it signals): arrive on the grid barrier, then wait
    // until every CTA has.  Warp 0 waits as a whole; the others wait at the
    // consumer barrier that staging opens with.
    __threadfence();
    consumer_sync(NCT);
    if (warp == 0) {
        if (lane == 0) {
            bool ok = mbar_wait_bounded(gready, 0u, P.timeout_ns);
            __threadfence();
            const uint32_t inc = bid == 0 ? 0x80000000u - (uint32_t)(grid - 1) : 1u;
            const uint32_t old = atomicAdd(P.gbar, inc);
            if (ok && N1 > 0) ok = grid_wait(P.gbar, old, P.timeout_ns);
            __threadfence();
            if (!ok) {
                record_status(P.status, STATUS_TIMEOUT);
                atomicExch(sm.abort_flag, 1);
            }
        }
        __syncwarp();
    }
    if (N1 > 0) {
        ffn_consume<F1, R1, true>(P, K, sm, P.geo[1], sm.segs[1], N1, NCT, red_tile, st);
        reduce_last(P1, NT, 1);
    }
}

}  // namespace

// Kernel: phase 0 of format F0 with R0-row items, phase 1 of F1 with R1.
template <int F0, int R0, int F1, int R1>
__global__ void __launch_bounds__(32 * (qmv_max_consumer_warps(R0 > R1 ? R0 : R1) + 1), 2)
    qmv_ffn_kernel(const __grid_constant__ QmvParams P, const GroupConsts K) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    const int S_ = P.nstages;
    const int Umax = max(P.geo[0].U, P.geo[1].U);
    const FfnSmem L = qmv_ffn_smem(Umax, P.red_tile, S_, P.stage_bytes);
    Smem sm;
    sm.stages = smem + L.stages;
    sm.xs = reinterpret_cast<float*>(smem + L.xs);
    sm.sxs = reinterpret_cast<float*>(smem + L.sxs);
    sm.red = reinterpret_cast<float*>(smem + L.red);
    sm.full = reinterpret_cast<uint64_t*>(smem + L.bars);
    sm.empty = sm.full + S_;
    sm.xfull = sm.empty + S_;
    uint64_t* gready = sm.xfull + 1;
    sm.cnt = reinterpret_cast<int*>(gready + 1);
    sm.abort_flag = sm.cnt + (S_ + 1);
    Seg* segs = reinterpret_cast<Seg*>(smem + L.segs);
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&P.seg[0]);
        uint32_t* dst = reinterpret_cast<uint32_t*>(segs);
        const int nw = 2 * (int)(sizeof(Seg) / 4);
        for (int i = threadIdx.x; i < nw; i += blockDim.x) dst[i] = src[i];
    }
    sm.segs = segs;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S_; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], (blockDim.x >> 5) - 1);
        }
        mbar_init(sm.xfull, 1);
        mbar_init(gready, 1);
        for (int s = 0; s <= S_; ++s) sm.cnt[s] = 0;
        *sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    qmv_ffn_cta<F0, R0, F1, R1>(P, K, sm, gready);
}

namespace {

// (gate/up format, down format) pairs with a one-launch kernel
template <int F0, int F1>
void* ffn_fn() {
    return reinterpret_cast<void*>(
        qmv_ffn_kernel<F0, qmv_rows_per_item(1, F0 == FMT_Q4_K ? 1 : F0 == FMT_Q6_K ? 2 : 4), F1,
                       qmv_rows_per_item(1, F1 == FMT_Q4_K ? 1 : F1 == FMT_Q6_K ? 2 : 4)>);
}

void* ffn_get(int f0, int f1) {
    if (f0 == FMT_Q4_K && f1 == FMT_Q6_K) return ffn_fn<FMT_Q4_K, FMT_Q6_K>();
    if (f0 == FMT_Q4_K && f1 == FMT_Q4_K) return ffn_fn<FMT_Q4_K, FMT_Q4_K>();
    if (f0 == FMT_Q6_K && f1 == FMT_Q6_K) return ffn_fn<FMT_Q6_K, FMT_Q6_K>();
    if (f0 == FMT_Q8_0 && f1 == FMT_Q8_0) return ffn_fn<FMT_Q8_0, FMT_Q8_0>();
    return nullptr;
}

}  // namespace

bool qmv_ffn_available(int f0, int f1) { return ffn_get(f0, f1) != nullptr; }

cudaError_t qmv_ffn_set_smem(int bytes) {
    const int pairs[4][2] = {{FMT_Q4_K, FMT_Q6_K}, {FMT_Q4_K, FMT_Q4_K}, {FMT_Q6_K, FMT_Q6_K}, {FMT_Q8_0, FMT_Q8_0}};
    for (auto& p : pairs) {
        cudaError_t e = cudaFuncSetAttribute(ffn_get(p[0], p[1]), cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t qmv_ffn_occupancy(int f0, int f1, int nt, size_t smem, int* per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, ffn_get(f0, f1), nt, smem);
}

// Launched with programmatic stream serialization, like the single-phase kernel.
cudaError_t qmv_ffn_launch(const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st) {
    const GroupConsts K = group_consts();
    void* args[2] = {const_cast<QmvParams*>(&P), const_cast<GroupConsts*>(&K)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(nt);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, ffn_get(P.fmt0, P.fmt1), args);
}

}  // namespace lq
