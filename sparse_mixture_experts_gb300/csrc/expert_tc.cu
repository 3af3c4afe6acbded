// expert_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05 + TMEM, operands staged by TMA), for token counts where every
// routed expert sees many rows (prefill).
//
// Per group g (a routed expert with n_g rows, or the shared expert with all T
// rows), rows taken in the expert-sorted order the grouping kernel produced
// ("Engine", Prefill: tokens grouped by expert, gathered, projected,
// scattered back):
//   gate/up GEMM : [gate | up] = Xp_g W^T over H, then h = act(gate, up)
//                  ("Llama Forward Pass", SwiGLU FFN; "Phase 19: MoE --
//                  gpt-oss-20b", section 2 Experts, with biases and clamps)
//   down GEMM    : y = h_g W_down^T over F (+ b_down), written as
//                  w_slot * y to the (token, slot) row of the combine buffer
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0    TMA producer: A (128 token rows) and B (N weight rows) tiles,
//             64 bf16 of K per stage, 128-byte swizzled, into an S-stage ring
//   warp 1    TMEM allocator and MMA issuer (one elected thread):
//             tcgen05.mma.cta_group::1.kind::f16, M=128, N=256 (expert
//             GEMMs; 128 for the router), K=16, fp32 accumulators in TMEM,
//             two accumulator buffers
//   warps 2-5 epilogue: tcgen05.ld of the accumulators, activation or
//             routing weight, stores
// Every mbarrier wait is bounded (about a second of %globaltimer); on
// timeout the kernel records an error in the status word, stops issuing
// work, waits (bounded) for its own copies and MMAs in flight, frees TMEM and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "lowbit.cuh"
#include "tc_ptx.cuh"

namespace moe {

constexpr int TC_THREADS = 192;
constexpr int A_TILE_BYTES = TC_BM * TC_BK * 2;        // 16 KB

// Per tile width BN (the MMA's N): the B tile, the stage, the ring depth and
// the TMEM columns (two accumulators of BN fp32 columns per M half).  N = 256
// halves the A bytes staged per weight byte, which matters because a CTA's TMA
// stream, not HBM, limits these GEMMs once the A rows are re-read from L2.
// Low-bit weights come in two shapes.  BN = 128: tiles of TC_LB_TM = 256 token
// rows, two M = 128 halves, each with its own MMA-issuing thread and
// accumulators, multiply the same widened B tile (one packed block), so that
// the widening -- the work that paces these kernels -- is done once per 256
// rows; for experts with more than 128 rows.  BN = 256: 128-row tiles against
// two packed blocks, half the stages (and their fixed costs) where the experts
// have fewer rows and the second half would stay empty.
template <int BN, int QF = QF_NONE>
struct TcShape {
    static constexpr bool LOWBIT = QF != QF_NONE;
    static constexpr int MH = LOWBIT && BN == TC_LB_BN ? TC_LB_TM / TC_BM : 1;  // M halves per tile
    static constexpr int NBLK = BN / 128;  // low-bit: packed blocks per stage
    static constexpr int BLK = QF == QF_Q4 ? LOWBIT_BLK_Q4 : LOWBIT_BLK_MXFP4;
    static constexpr int A_BYTES = MH * A_TILE_BYTES;
    static constexpr int B_BYTES = BN * TC_BK * 2;
    static constexpr int STAGE = (A_BYTES + B_BYTES + 1023) / 1024 * 1024;
    static constexpr int STAGES = LOWBIT ? (MH == 2 ? 4 : 3) : (BN == 256 ? 4 : 6);
    // low-bit weights: the packed blocks (codes and scales of 128 rows x 64 K
    // each) of each stage's B tile land in a ring of their own, filled ahead
    // of the A/B ring, from which dequantising warps write the bf16 B tile
    static constexpr int RAW_STAGE = LOWBIT ? NBLK * BLK : 0;
    static constexpr int RAW_STAGES = LOWBIT ? 4 : 0;
    static constexpr int RAW_OFF = STAGES * STAGE;
    static constexpr int BAR_OFF = RAW_OFF + (RAW_STAGES * RAW_STAGE + 1023) / 1024 * 1024;
    static constexpr int TMEM_COLS = 2 * MH * BN;
    // after the rings: barriers, then the epilogue's staging (4 warps x 32 rows
    // x 16 fp32), then (MXFP4) the conversion tables of the 256 scale bytes
    static constexpr int STAGING_OFF = BAR_OFF + 512;
    static constexpr int STAGING_BYTES = 4 * 32 * 16 * 4;
    static constexpr int TAB_OFF = STAGING_OFF + STAGING_BYTES;
    static constexpr int TAB_BYTES = QF == QF_MXFP4 ? 256 * (int)sizeof(Fp4Table) : 0;
    static constexpr size_t SMEM = (size_t)TAB_OFF + TAB_BYTES + 1024 /*align*/;
    // dequantising warps: one (B row, K half) per thread (BN = 128), or one B row (BN = 256)
    static constexpr int DQ_THREADS = LOWBIT ? 256 : 0;
    static constexpr int RAW_WARP = (TC_THREADS + DQ_THREADS) / 32;  // the raw ring's producer (low-bit)
    static constexpr int MMA2_WARP = RAW_WARP + 1;                   // the second M half's MMA issuer (MH = 2)
    static constexpr int THREADS = TC_THREADS + DQ_THREADS + (LOWBIT ? 32 * MH : 0);
    // tile geometry (tc_geometry gives the same to the grouping kernel)
    static constexpr int TM = MH * TC_BM;
    // barriers: full, empty, bready per A/B stage; two accumulators' full and
    // empty; a drain per M half; raw full and empty per raw stage; the TMEM
    // address and the abort word
    static_assert((3 * STAGES + 6 + 2 * RAW_STAGES) * 8 + 8 <= 512, "barrier area");
    static_assert(TMEM_COLS <= 512, "tensor memory");
    static_assert(SMEM <= 232448, "shared memory per block");
    static_assert(!LOWBIT || BN == 128 || BN == 256, "low-bit tiles are one or two packed blocks wide");
};

struct TensorMaps {
    CUtensorMap xp;       // A of gate/up: [Tmax*K + Tmax][H]
    CUtensorMap h;        // A of down:    [Tmax*K + Tmax][Fmax]
    CUtensorMap gate;     // [E*F][H], box TC_BN_UP / 2 rows
    CUtensorMap up;       // [E*F][H]
    CUtensorMap down;     // [E*H][F], box TC_BN_DOWN rows
    CUtensorMap sh_gate;  // [Fs][H]
    CUtensorMap sh_up;    // [Fs][H]
    CUtensorMap sh_down;  // [H][Fs]
    CUtensorMap router;   // [R][H], box 128 rows
};

// A operand, then the B operand(s) of the routed experts and of the shared
// expert; the gate/up GEMM loads two B boxes of TC_BN_UP / 2 rows (gate rows,
// up rows), the down GEMM one box of TC_BN_DOWN rows (b1 / sb1 unused), the
// router GEMM one of 128 rows.
struct TcMaps {
    CUtensorMap a, b0, b1, sb0, sb1;
    CUtensorMap sa;  // A of the shared expert's gate/up tiles: x itself (its rows are all tokens in order)
};

// ---------------------------------------------------------------------------
// the grouped GEMM kernel
// ---------------------------------------------------------------------------
enum { EPI_UP = 0, EPI_DOWN = 1, EPI_ROUTER = 2 };

struct TcArgs {
    const int *gfirst;  // first tile of each group and the total (this GEMM's order)
    const int *active;  // routed experts with tokens, ascending
    const RouteMeta *meta;
    const int *counts, *offsets, *expert_rows;
    const float *gate_b, *up_b, *down_b;
    const float *topk_w, *sh_gate;
    __nv_bfloat16 *h;   // EPI_UP output
    float *ys;          // EPI_DOWN output: weighted per-slot outputs [T][K+1][H], fp32
    float *logits;      // EPI_ROUTER output [T][R] (router_S == 1)
    float *rparts;      // EPI_ROUTER output [router_S][T][R] partial sums over K ranges (router_S > 1)
    const float *router_b;
    int R, router_nt, router_S, router_bn;  // router rows, router N tiles, K splits, tile width
    int *status;
    const uint8_t *fp4;          // low-bit weights: packed blocks of gate/up ([E][F/64][H/64]) or down ([E][H/128][F/64])
    const volatile int *stall;   // test-only fault injection: a word nothing sets, waited for (else null)
    unsigned long long wait_ns;  // bound of that wait
    int T, K, E, H, F, Fs, Fmax, Tmax;
    int act;
    float alpha, limit;
};

struct TileInfo {
    int g, m0, n0;
    int rows;     // rows of the group
    int a_row0;   // first row of the group in the A tensor
    int kb0, nk;  // first K block, K blocks
    int split;    // router: K range of the tile
    bool shared;
};

// group tables of this launch (global memory, written by the grouping kernel
// before the launch; read through the read-only path): first tile of each
// group (and the total), each group's expert (E for the shared expert), its
// rows and its first row in the expert-sorted buffers
struct GroupTab {
    const int *first;
    const int *expert;
    const int *rows, *row0;
    int n;
};

// gcur: the caller's group cursor (each role visits its tiles in increasing
// order, so the group only moves forward); start at 0
template <int EPI, int TM, int TNU, int TND>
__device__ __forceinline__ bool tile_info(const TcArgs &a, int t, TileInfo &ti, const GroupTab &gt, int &gcur)
{
    if (EPI == EPI_ROUTER) {
        // dense: every 128-token tile against every 128-row tile of the router,
        // K split in router_S ranges (so that the small GEMM covers the GPU)
        const int per = a.router_nt * a.router_S;
        const int rem = t % per;
        ti.g = 0;
        ti.m0 = (t / per) * TC_BM;
        ti.n0 = (rem / a.router_S) * a.router_bn;
        ti.split = rem % a.router_S;
        ti.shared = false;
        ti.rows = a.T;
        ti.a_row0 = 0;
        const int nkb = a.H / TC_BK;
        ti.kb0 = nkb * ti.split / a.router_S;
        ti.nk = nkb * (ti.split + 1) / a.router_S - ti.kb0;
        return ti.nk > 0;
    }
    ti.kb0 = 0;
    ti.split = 0;
    // the group of tile t: the last one whose first tile is <= t; within a
    // group the tiles run (n, m) with m fastest
    if (gt.n <= 0 || t < 0 || t >= __ldg(gt.first + gt.n)) return false;
    int lo = gcur;
    if (lo < 0 || lo >= gt.n || __ldg(gt.first + lo) > t || __ldg(gt.first + lo + 1) <= t) {
        // binary search (every group has a tile, so first[] increases strictly
        // from first[0] = 0)
        int l = 0, h = gt.n - 1;
        while (l < h) {
            const int m = (l + h + 1) >> 1;
            if (__ldg(gt.first + m) <= t) l = m;
            else h = m - 1;
        }
        lo = l;
    }
    gcur = lo;
    ti.g = __ldg(gt.expert + lo);
    ti.shared = ti.g == a.E;
    if (ti.g < 0 || ti.g > a.E || (ti.shared && a.Fs == 0)) return false;
    ti.rows = __ldg(gt.rows + lo);
    ti.a_row0 = __ldg(gt.row0 + lo);
    const int mt = (ti.rows + TM - 1) / TM;
    if (mt <= 0) return false;
    const int local = t - __ldg(gt.first + lo);
    const int n = local / mt;
    ti.m0 = (local - n * mt) * TM;
    ti.n0 = n * (EPI == EPI_UP ? TNU : TND);
    if (EPI == EPI_UP) ti.nk = a.H / TC_BK;
    else ti.nk = (ti.shared ? a.Fs : a.F) / TC_BK;
    return ti.m0 >= 0 && ti.m0 < ti.rows && ti.n0 >= 0;
}

// 16 consecutive fp32 biases (zeros for a layer without them); p is 16-byte aligned
__device__ __forceinline__ void bias16(const float *p, float (&b)[16])
{
    if (p) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p) + q);
            b[4 * q] = v.x; b[4 * q + 1] = v.y; b[4 * q + 2] = v.z; b[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i] = 0.0f;
    }
}

// 16 (gate, up) accumulator pairs plus their biases through the activation,
// packed as 8 bf16 pairs (feature 2i in the low half)
template <int ACT>
__device__ __forceinline__ void glu_pack16(const uint32_t (&g)[16], const uint32_t (&u)[16], const float (&gb)[16],
                                           const float (&ub)[16], float alpha, float limit, uint32_t (&packed)[8])
{
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float v0 = activation<ACT>(__uint_as_float(g[i]) + gb[i], __uint_as_float(u[i]) + ub[i], alpha, limit);
        const float v1 =
            activation<ACT>(__uint_as_float(g[i + 1]) + gb[i + 1], __uint_as_float(u[i + 1]) + ub[i + 1], alpha, limit);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(v0, v1);
        packed[i / 2] = *reinterpret_cast<uint32_t *>(&p2);
    }
}

template <int EPI, int BN, typename Maps, int QF = QF_NONE>
__global__ void __launch_bounds__(TcShape<BN, QF>::THREADS, 1) tc_gemm_kernel(const __grid_constant__ Maps maps,
                                                                               const TcArgs a)
{
    using Sh = TcShape<BN, QF>;
    constexpr bool FP4 = Sh::LOWBIT;
    constexpr int LB_BLK = Sh::BLK;
    constexpr int TC_STAGES = Sh::STAGES;
    constexpr int STAGE_BYTES = Sh::STAGE;
    constexpr int B_TILE_BYTES = Sh::B_BYTES;
    constexpr int TMEM_COLS = Sh::TMEM_COLS;
    constexpr int MH = Sh::MH;
    constexpr int TNU = BN / 2;  // gate/up features per tile
    constexpr int TND = BN;      // down output columns per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Sh::BAR_OFF);
    uint64_t *empty = full + TC_STAGES;
    uint64_t *acc_full = empty + TC_STAGES;   // [2]
    uint64_t *acc_empty = acc_full + 2;       // [2]
    uint64_t *drain = acc_empty + 2;          // [2] each MMA thread's own completion, after an abort
    uint64_t *bready = drain + 2;             // [TC_STAGES] low-bit weights: the B tile is dequantised
    uint64_t *raw_full = bready + TC_STAGES;  // [RAW_STAGES] low-bit weights: the packed blocks landed
    uint64_t *raw_empty = raw_full + Sh::RAW_STAGES;  // [RAW_STAGES] ... and were read
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(raw_empty + Sh::RAW_STAGES);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = EPI == EPI_ROUTER ? ((a.T + TC_BM - 1) / TC_BM) * a.router_nt * a.router_S
                                          : (EPI == EPI_UP ? a.meta->n_up_tiles : a.meta->n_down_tiles);

    if (threadIdx.x == 0) {
        // empty and acc_full: one arrival per M half's MMA thread
        for (int s = 0; s < TC_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], MH);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], MH);
            mbar_init(&acc_empty[b], 128);
            mbar_init(&drain[b], 1);
        }
        if (FP4) {
            for (int st = 0; st < TC_STAGES; ++st) mbar_init(&bready[st], Sh::DQ_THREADS);
            for (int st = 0; st < Sh::RAW_STAGES; ++st) {
                mbar_init(&raw_full[st], 1);
                mbar_init(&raw_empty[st], Sh::DQ_THREADS);
            }
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    GroupTab gt{nullptr, nullptr, nullptr, nullptr, 0};
    int gcur = 0;  // this thread's group cursor
    if constexpr (EPI != EPI_ROUTER) {
        const int P = a.E + 2;
        gt.first = a.gfirst + (EPI == EPI_UP ? 0 : P);
        gt.expert = a.gfirst + 2 * P;
        gt.rows = a.gfirst + 3 * P;
        gt.row0 = a.gfirst + 4 * P;
        gt.n = a.meta->n_active + (a.Fs > 0 ? 1 : 0);
    }
    Fp4Table *fp4tab = reinterpret_cast<Fp4Table *>(smem + Sh::TAB_OFF);
    if constexpr (QF == QF_MXFP4)
        for (int i = threadIdx.x; i < 256; i += Sh::THREADS) fp4tab[i] = mxfp4_table((uint32_t)i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            tmap_prefetch(&maps.a);
            if (EPI == EPI_UP) tmap_prefetch(&maps.sa);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t used = 0, last_phase = 0;  // per stage: loads issued, parity of the last
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                TileInfo ti;
                if (!tile_info<EPI, Sh::TM, TNU, TND>(a, t, ti, gt, gcur)) {
                    record_error(a.status, DEV_BAD_TILE);
                    *abort_flag = 1;
                    break;
                }
                for (int kb = 0; kb < ti.nk; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
                        record_error(a.status, DEV_TIMEOUT_EMPTY_BARRIER);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + stage * STAGE_BYTES;
                    uint8_t *sb = sa + A_TILE_BYTES;
                    const int kc = (ti.kb0 + kb) * TC_BK;
                    if constexpr (FP4) {
                        // the A tiles only (rows m0 .. m0+127, and m0+128 .. m0+255 where
                        // the group has such rows): the raw ring's producer copies the
                        // packed weight block, and the dequantising warps write the B tile
                        const bool two = MH == 2 && ti.m0 + TC_BM < ti.rows;
                        mbar_arrive_expect_tx(&full[stage], two ? 2 * A_TILE_BYTES : A_TILE_BYTES);
                        tma_load_2d(sa, &maps.a, &full[stage], kc, ti.a_row0 + ti.m0);
                        if (two) tma_load_2d(sa + A_TILE_BYTES, &maps.a, &full[stage], kc, ti.a_row0 + ti.m0 + TC_BM);
                        used |= 1u << stage;
                        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                        if (++stage == TC_STAGES) stage = 0, phase ^= 1;
                        continue;
                    }
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    if (EPI == EPI_UP && ti.shared) tma_load_2d(sa, &maps.sa, &full[stage], kc, ti.m0);
                    else tma_load_2d(sa, &maps.a, &full[stage], kc, ti.a_row0 + ti.m0);
                    if (EPI == EPI_UP) {
                        const int brow = ti.shared ? ti.n0 : ti.g * a.F + ti.n0;
                        tma_load_2d(sb, ti.shared ? &maps.sb0 : &maps.b0, &full[stage], kc, brow);
                        tma_load_2d(sb + B_TILE_BYTES / 2, ti.shared ? &maps.sb1 : &maps.b1, &full[stage], kc, brow);
                    } else {
                        const int brow = ti.shared ? ti.n0 : ti.g * a.H + ti.n0;
                        tma_load_2d(sb, ti.shared ? &maps.sb0 : &maps.b0, &full[stage], kc, brow);
                    }
                    used |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == TC_STAGES) stage = 0, phase ^= 1;
                }
            }
            // drain: no copy of ours may still be landing when the CTA exits
            volatile int never = 0;
            for (int s = 0; s < TC_STAGES; ++s)
                if ((used >> s) & 1u) mbar_wait(&full[s], (last_phase >> s) & 1u, &never);
        }
    } else if (warp == 1 || (MH == 2 && warp == Sh::MMA2_WARP)) {
        // ------------------------------ MMA issuers ------------------------------
        // One thread per M half (low-bit tiles have two): half h multiplies the
        // A rows m0 + 128h .. m0 + 128h + 127 with the stage's B tile into its
        // own accumulator columns.  A half without rows in the tile issues
        // nothing and arrives on the barriers its MMAs would have signalled.
        if (lane == 0) {
            const int half = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            bool issued = false;  // any MMA of this thread
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++it) {
                TileInfo ti;
                if (!tile_info<EPI, Sh::TM, TNU, TND>(a, t, ti, gt, gcur)) break;
                const int b = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(&acc_empty[b], acc_phase ^ 1, abort_flag)) {
                    record_error(a.status, DEV_TIMEOUT_ACCUM_FREE);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const bool active = ti.m0 + half * TC_BM < ti.rows;
                const uint32_t d_tmem = tmem_base + (uint32_t)((b * MH + half) * BN);
                for (int kb = 0; kb < ti.nk; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag) ||
                        (FP4 && !mbar_wait(&bready[stage], phase, abort_flag))) {
                        record_error(a.status, DEV_TIMEOUT_FULL_BARRIER);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (active) {
                        const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES) + half * A_TILE_BYTES;
                        const uint32_t sb = smem_u32(smem + stage * STAGE_BYTES) + Sh::A_BYTES;
#pragma unroll
                        for (int k = 0; k < TC_BK / 16; ++k) {
                            // advance 16 bf16 = 32 bytes along K inside the swizzled row
                            mma_bf16(d_tmem, smem_desc_sw128(sa + k * 32), smem_desc_sw128(sb + k * 32), idesc,
                                     (kb | k) != 0);
                        }
                        mma_commit(&empty[stage]);
                        issued = true;
                    } else {
                        mbar_arrive(&empty[stage]);
                    }
                    if (++stage == TC_STAGES) stage = 0, phase ^= 1;
                }
                if (!ok) break;
                if (active) mma_commit(&acc_full[b]);
                else mbar_arrive(&acc_full[b]);
            }
            // every MMA this thread issued completes before the shared memory it
            // reads and the tensor memory it writes are released: after an abort
            // the epilogue may not wait for the accumulators (and a tile's last
            // MMAs may not be committed to one)
            if (issued) {
                volatile int never = 0;
                mma_commit(&drain[half]);
                mbar_wait(&drain[half], 0, &never);
            }
        }
    } else if (FP4 && warp == Sh::RAW_WARP) {
        // ------------------------------ raw ring producer (low-bit, last warp) ------------------------------
        // The packed blocks of each stage's BN weight rows (gate/up: per block 64
        // features as 64 gate + 64 up rows; down: 128 output rows), in the A/B
        // ring's order; a block past the matrix is not copied (its rows are
        // written as zeros).
        if (lane == 0) {
            int rs = 0;
            uint32_t rph = 0;
            uint32_t used = 0, last_phase = 0;  // per raw stage: copies issued, parity of the last
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                TileInfo ti;
                if (!tile_info<EPI, Sh::TM, TNU, TND>(a, t, ti, gt, gcur)) break;  // the A producer records it
                const int nb = EPI == EPI_UP ? a.F / 64 : (a.H + 127) / 128;
                const int b0 = EPI == EPI_UP ? ti.n0 / 64 : ti.n0 / 128;  // < nb
                const int nvalid = min(Sh::NBLK, nb - b0);
                const int nkbt = EPI == EPI_UP ? a.H / TC_BK : a.F / TC_BK;
                for (int kb = 0; kb < ti.nk; ++kb) {
                    if (!mbar_wait(&raw_empty[rs], rph ^ 1, abort_flag)) {
                        record_error(a.status, DEV_TIMEOUT_EMPTY_BARRIER);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    uint8_t *dst = smem + Sh::RAW_OFF + rs * Sh::RAW_STAGE;
                    mbar_arrive_expect_tx(&raw_full[rs], nvalid * LB_BLK);
                    for (int q = 0; q < nvalid; ++q) {
                        const size_t blk = ((size_t)ti.g * nb + b0 + q) * nkbt + ti.kb0 + kb;
                        bulk_load(dst + q * LB_BLK, a.fp4 + blk * LB_BLK, LB_BLK, &raw_full[rs]);
                    }
                    used |= 1u << rs;
                    last_phase = (last_phase & ~(1u << rs)) | (rph << rs);
                    if (++rs == Sh::RAW_STAGES) rs = 0, rph ^= 1;
                }
            }
            // drain: no copy of ours may still be landing when the CTA exits
            volatile int never = 0;
            for (int st = 0; st < Sh::RAW_STAGES; ++st)
                if ((used >> st) & 1u) mbar_wait(&raw_full[st], (last_phase >> st) & 1u, &never);
        }
    } else if (FP4 && warp >= 6) {
        // ------------------------------ low-bit dequantisation (warps 6..13) ------------------------------
        // Per stage: the rows of the B tile, in their 128-byte-swizzled layout
        // (chunk c of row r at r * 128 + ((c ^ (r & 7)) << 4), the layout the TMA
        // would have written).  BN = 128: the 128 rows of the stage's packed
        // block, in order, each K half of a row by one thread (32 codes, four
        // chunks).  BN = 256: one row per thread (64 codes, eight chunks) from
        // two blocks (gate/up: B rows 0..127 are the gate rows of features
        // n0 .. n0+127, 128..255 the up rows, block q holding features 64q ..
        // 64q+63 as 64 gate then 64 up rows; down: block q holds B rows 128q ..
        // 128q+127); a block past the matrix gives zero rows.  A thread loads
        // its codes and scales from the raw ring, waits until the MMAs have
        // finished with the A/B stage, widens the codes to bf16 (MXFP4 exactly,
        // Q4 rounded once) and writes them; then the writes are made visible to
        // the tensor cores' reads, the stage is released to the MMAs and the raw
        // stage to its producer.
        const int dq = threadIdx.x - TC_THREADS;  // 0 .. 255
        const int rr = MH == 2 ? dq & 127 : dq;   // the B-tile row of this thread
        const int hk = MH == 2 ? dq >> 7 : 0;     // its K half (BN = 128)
        int q = 0, brow = rr;                     // its packed block and the row in it
        if (MH == 1) {
            if (EPI == EPI_UP) {
                const int f = rr & 127;
                q = f >> 6;
                brow = (rr < 128 ? 0 : 64) + (f & 63);
            } else {
                q = rr >> 7;
                brow = rr & 127;
            }
        }
        int stage = 0, rs = 0;
        uint32_t phase = 0, rph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            TileInfo ti;
            if (!tile_info<EPI, Sh::TM, TNU, TND>(a, t, ti, gt, gcur)) break;
            const int nb = EPI == EPI_UP ? a.F / 64 : (a.H + 127) / 128;
            const int b0 = EPI == EPI_UP ? ti.n0 / 64 : ti.n0 / 128;
            const bool zero = b0 + q >= nb;
            for (int kb = 0; kb < ti.nk; ++kb) {
                if (!mbar_wait(&raw_full[rs], rph, abort_flag)) {
                    record_error(a.status, DEV_TIMEOUT_FULL_BARRIER);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                const uint8_t *blk = smem + Sh::RAW_OFF + rs * Sh::RAW_STAGE + q * LB_BLK;
                LowbitHalf xh;
                LowbitRow xr;
                if (MH == 2) lowbit_load_half<QF>(blk, rr, hk, xh);
                else if (!zero) lowbit_load_row<QF>(blk, brow, xr);
                const int rs_read = rs;  // released after the proxy fence below
                if (++rs == Sh::RAW_STAGES) rs = 0, rph ^= 1;
                if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
                    record_error(a.status, DEV_TIMEOUT_EMPTY_BARRIER);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                uint4 *dst = reinterpret_cast<uint4 *>(smem + stage * STAGE_BYTES + Sh::A_BYTES + rr * 128);
                if (MH == 2) {
                    uint32_t v[16];
                    lowbit_widen_half<QF>(xh, fp4tab, v);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[(4 * hk + j) ^ (rr & 7)] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                } else if (zero) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) dst[j ^ (rr & 7)] = make_uint4(0, 0, 0, 0);
                } else {
                    uint32_t v[32];
                    lowbit_widen_row<QF>(xr, fp4tab, v);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j ^ (rr & 7)] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
                // one proxy fence orders this thread's B-tile writes before the MMAs'
                // reads and its raw-stage reads before the bulk copy that refills
                // the stage (both async proxy): the barriers alone do not order
                // generic accesses with async-proxy ones (without the fence on the
                // raw reads the copy could land in rows still being read, which
                // showed as nondeterministic weight rows)
                fence_proxy_async_shared();
                mbar_arrive(&bready[stage]);
                mbar_arrive(&raw_empty[rs_read]);
                if (++stage == TC_STAGES) stage = 0, phase ^= 1;
            }
        }
    } else {
        // ------------------------------ epilogue (warps 2..5) ------------------------------
        const int q = warp & 3;             // TMEM lane quarter this warp may access
        const int r = q * 32 + lane;        // accumulator row (tile row) of this thread
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        int it = 0;
        bool run = true;
        if (a.stall) {
            // test-only fault injection: every epilogue thread waits (bounded) for
            // a word that nothing sets; when the wait runs out the CTA aborts
            // with the MMA and the copies in flight, which then drain
            const unsigned long long t0 = globaltimer();
            while (*a.stall == 0) {
                __nanosleep(256);
                if (*abort_flag || globaltimer() - t0 > a.wait_ns) break;
            }
            if (*a.stall == 0) {
                record_error(a.status, DEV_TIMEOUT_INJECTED);
                *abort_flag = 1;
                run = false;
            }
        }
        for (int t = blockIdx.x; run && t < n_tiles; t += gridDim.x, ++it) {
            TileInfo ti;
            if (!tile_info<EPI, Sh::TM, TNU, TND>(a, t, ti, gt, gcur)) break;
            const int b = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            // gate/up: the tile's gate and up biases (lane l: features 4l .. 4l+3),
            // loaded before the accumulator wait so that their latency is hidden
            float4 bgl = make_float4(0.0f, 0.0f, 0.0f, 0.0f), bul = bgl;
            if (EPI == EPI_UP && !ti.shared && 4 * lane < min(BN / 2, a.F - ti.n0)) {
                const size_t o = (size_t)ti.g * a.F + ti.n0 + 4 * lane;
                if (a.gate_b) bgl = __ldg(reinterpret_cast<const float4 *>(a.gate_b + o));
                if (a.up_b) bul = __ldg(reinterpret_cast<const float4 *>(a.up_b + o));
            }
            if (!mbar_wait(&acc_full[b], acc_phase, abort_flag)) {
                record_error(a.status, DEV_TIMEOUT_ACCUM_BARRIER);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            if (EPI == EPI_UP) {
                // the biases through this warp's staging area: [gate 128][up 128]
                float4 *bs = reinterpret_cast<float4 *>(smem + Sh::STAGING_OFF) + q * 128;
                __syncwarp();  // the previous tile's reads are done
                bs[lane] = bgl;
                bs[32 + lane] = bul;
                __syncwarp();
            }
            // each M half of the tile that has rows (low-bit tiles have two)
            for (int hm = 0; hm < MH; ++hm) {
                if (ti.m0 + hm * TC_BM >= ti.rows) break;  // the same for the whole CTA
                const uint32_t tbase = tmem_base + lane_addr + (uint32_t)((b * MH + hm) * BN);
                const int j = ti.m0 + hm * TC_BM + r;  // row within the group
                const bool valid = j < ti.rows;
                if (EPI == EPI_ROUTER) {
                    // logits[t][n] (+ router bias), fp32, or with K split the partial
                    // sum of this K range (the bias in the first); R need not be a
                    // multiple of 4.  Each 32-row x 16-column chunk of the warp goes
                    // through its staging area (the layout of the down epilogue), so
                    // that a store instruction writes 2 rows x 16 consecutive logits
                    // instead of one logit in each of 32 rows.
                    float *dst = a.router_S > 1 ? a.rparts + (size_t)ti.split * a.T * a.R : a.logits;
                    const bool with_bias = a.router_b && ti.split == 0;
                    float4 *stg = reinterpret_cast<float4 *>(smem + Sh::STAGING_OFF) + q * 128;
                    const float *stf = reinterpret_cast<const float *>(stg);
                    const int cc = lane & 15;  // the column this lane stores
#pragma unroll 1
                    for (int c = 0; c < BN; c += 16) {
                        if (ti.n0 + c >= a.R) break;  // the same for the whole warp
                        uint32_t v[16];
                        tmem_ld16(tbase + c, v);
                        const int n = ti.n0 + c + cc;
                        const float b = (with_bias && n < a.E) ? a.router_b[n] : 0.0f;
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            stg[lane * 4 + (i ^ ((lane >> 1) & 3))] =
                                make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                            __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                        __syncwarp();
#pragma unroll 4
                        for (int it = 0; it < 16; ++it) {
                            const int rr = 2 * it + (lane >> 4);  // row of the warp's 32
                            const float val = stf[(rr * 4 + ((cc >> 2) ^ ((rr >> 1) & 3))) * 4 + (cc & 3)];
                            const int jr = ti.m0 + hm * TC_BM + q * 32 + rr;
                            if (jr < ti.rows && n < a.R) dst[(size_t)jr * a.R + n] = val + b;
                        }
                        __syncwarp();
                    }
                } else if (EPI == EPI_UP) {
                    const int fd = ti.shared ? a.Fs : a.F;
                    const int hcols = min(BN / 2, fd - ti.n0);  // a multiple of 64 (fd is)
                    __nv_bfloat16 *hrow = a.h + (size_t)(ti.a_row0 + j) * a.Fmax + ti.n0;
                    const bool swiglu = ti.shared || a.act == MOE_ACT_SWIGLU;
                    const float4 *bs = reinterpret_cast<const float4 *>(smem + Sh::STAGING_OFF) + q * 128;
#pragma unroll 1
                    for (int c = 0; c < BN / 2; c += 16) {
                        if (c >= hcols) break;
                        uint32_t g[16], u[16];
                        tmem_ld16(tbase + c, g);
                        tmem_ld16(tbase + BN / 2 + c, u);
                        float gb[16], ub[16];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float4 x = bs[c / 4 + k], y = bs[32 + c / 4 + k];
                            gb[4 * k] = x.x; gb[4 * k + 1] = x.y; gb[4 * k + 2] = x.z; gb[4 * k + 3] = x.w;
                            ub[4 * k] = y.x; ub[4 * k + 1] = y.y; ub[4 * k + 2] = y.z; ub[4 * k + 3] = y.w;
                        }
                        tmem_ld_wait();
                        uint32_t packed[8];
                        if (swiglu) glu_pack16<MOE_ACT_SWIGLU>(g, u, gb, ub, a.alpha, a.limit, packed);
                        else glu_pack16<MOE_ACT_CLAMP_GLU>(g, u, gb, ub, a.alpha, a.limit, packed);
                        if (valid) {
                            uint4 *dst = reinterpret_cast<uint4 *>(hrow + c);
                            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                        }
                    }
                } else {
                    int tok = 0, slot = 0;
                    float wgt = 0.0f;
                    if (valid) {
                        if (ti.shared) { tok = j; slot = a.K; wgt = a.sh_gate[tok]; }
                        else {
                            const int p = a.expert_rows[ti.a_row0 + j];
                            tok = p / a.K; slot = p - tok * a.K; wgt = a.topk_w[p];
                        }
                    }
                    const float *bd = (!ti.shared && a.down_b) ? a.down_b + (size_t)ti.g * a.H + ti.n0 : nullptr;
                    // this thread's fp32 row of the per-slot buffer (0: a row past the group's end)
                    const unsigned long long yrow =
                        valid ? reinterpret_cast<unsigned long long>(a.ys + ((size_t)tok * (a.K + 1) + slot) * a.H + ti.n0)
                              : 0ull;
                    const int ncols = min(BN, a.H - ti.n0);  // the same for the whole tile; a multiple of 64 (H is)
                    // Each thread holds one row; the warp's 32 rows x 16 columns go
                    // through shared memory so that each store instruction writes 8
                    // rows x 64 contiguous bytes (whole sectors) instead of 32 rows x
                    // 16 bytes.  Row r's float4 q sits at r * 4 + (q ^ ((r >> 1) & 3)):
                    // no bank conflicts for the row-wise writes or the column-wise reads.
                    float4 *stg = reinterpret_cast<float4 *>(smem + Sh::STAGING_OFF) + q * 128;
#pragma unroll 1
                    for (int c = 0; c < ncols; c += 16) {
                        uint32_t v[16];
                        tmem_ld16(tbase + c, v);
                        float bb[16];
                        bias16(bd ? bd + c : nullptr, bb);
                        tmem_ld_wait();
                        float o[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = wgt * (__uint_as_float(v[i]) + bb[i]);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            stg[lane * 4 + (i ^ ((lane >> 1) & 3))] =
                                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int f = i * 32 + lane, rr = f >> 2, qq = f & 3;
                            const float4 val = stg[rr * 4 + (qq ^ ((rr >> 1) & 3))];
                            const unsigned long long dst = __shfl_sync(0xffffffffu, yrow, rr);
                            if (dst) reinterpret_cast<float4 *>(reinterpret_cast<float *>(dst) + c)[qq] = val;
                        }
                        __syncwarp();
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows][inner], row pitch = inner elements, box = 64 x box_rows, 128-byte swizzle
static bool encode_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)TC_BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_supported(const Layer &L, std::string &why)
{
    if (L.cfg.w_dtype != MOE_DT_BF16) { why = "tensor-core path needs bf16 weights"; return false; }
    if (L.H % 64 || L.F % 64 || L.Fs % 64) { why = "tensor-core path needs H, F, Fs multiples of 64"; return false; }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, L.device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, L.device);
    if (major != 10 || minor != 3) { why = "tensor-core kernels are built for sm_103a"; return false; }
    if (!get_encode()) { why = "cuTensorMapEncodeTiled unavailable"; return false; }
    return true;
}


template <int EPI, int BN, int QF>
static bool set_smem()
{
    return cudaFuncSetAttribute(tc_gemm_kernel<EPI, BN, TcMaps, QF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)TcShape<BN, QF>::SMEM) == cudaSuccess;
}

// both tile shapes of both low-bit GEMMs
template <int QF>
static bool lowbit_smem()
{
    return set_smem<EPI_UP, TC_LB_BN, QF>() && set_smem<EPI_DOWN, TC_LB_BN, QF>() && set_smem<EPI_UP, 256, QF>() &&
           set_smem<EPI_DOWN, 256, QF>();
}

template <int EPI, int QF>
static void launch_lowbit(const TcMaps &maps, const TcArgs &a, bool two_halves, int grid, cudaStream_t s)
{
    if (two_halves) {
        using Sh = TcShape<TC_LB_BN, QF>;
        tc_gemm_kernel<EPI, TC_LB_BN, TcMaps, QF><<<grid, Sh::THREADS, Sh::SMEM, s>>>(maps, a);
    } else {
        using Sh = TcShape<256, QF>;
        tc_gemm_kernel<EPI, 256, TcMaps, QF><<<grid, Sh::THREADS, Sh::SMEM, s>>>(maps, a);
    }
}

int tc_prepare(Layer &L)
{
    TensorMaps *m = new (std::nothrow) TensorMaps();
    if (!m) return -1;
    const uint64_t rows_all = (uint64_t)L.Tmax * L.K + L.Tmax;
    bool ok = encode_2d(&m->xp, L.xp, L.H, rows_all, TC_BM) && encode_2d(&m->h, L.h, L.Fmax, rows_all, TC_BM) &&
              encode_2d(&m->router, L.router_w, L.H, (uint64_t)L.R, 128);
    if (L.qfmt != QF_NONE) {
        // the experts' B operand is dequantised from the packed blocks in the kernel
        m->gate = m->up = m->down = m->router;
    } else {
        // (the weight arrays hold wslots experts: every one, or the resident slots, a
        // layer that never runs these GEMMs)
        ok = ok && encode_2d(&m->gate, L.gate_w, L.H, (uint64_t)L.wslots * L.F, TC_BN_UP / 2) &&
             encode_2d(&m->up, L.up_w, L.H, (uint64_t)L.wslots * L.F, TC_BN_UP / 2) &&
             encode_2d(&m->down, L.down_w, L.F, (uint64_t)L.wslots * L.H, TC_BN_DOWN);
    }
    if (ok && L.Fs) {
        ok = encode_2d(&m->sh_gate, L.sh_gate_w, L.H, L.Fs, TC_BN_UP / 2) &&
             encode_2d(&m->sh_up, L.sh_up_w, L.H, L.Fs, TC_BN_UP / 2) &&
             encode_2d(&m->sh_down, L.sh_down_w, L.Fs, L.H, TC_BN_DOWN);
    } else if (ok) {
        m->sh_gate = m->gate;
        m->sh_up = m->up;
        m->sh_down = m->down;
    }
    if (!ok) { delete m; return -1; }
    if (cudaFuncSetAttribute(tc_gemm_kernel<EPI_UP, TC_BN_UP, TcMaps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)TcShape<TC_BN_UP>::SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<EPI_DOWN, TC_BN_DOWN, TcMaps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)TcShape<TC_BN_DOWN>::SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(tc_gemm_kernel<EPI_ROUTER, 128, TcMaps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)TcShape<128>::SMEM) != cudaSuccess ||
        !lowbit_smem<QF_MXFP4>() || !lowbit_smem<QF_Q4>()) {
        delete m;
        return -1;
    }
    L.tmaps = m;
    return 0;
}

void tc_release(Layer &L)
{
    delete L.tmaps;
    L.tmaps = nullptr;
}

static TcArgs make_tc_args(const Layer &L, int T)
{
    TcArgs a;
    a.meta = L.meta;
    a.counts = L.counts; a.offsets = L.offsets; a.expert_rows = L.expert_rows;
    a.gfirst = L.gfirst; a.active = L.active;
    a.gate_b = L.gate_b; a.up_b = L.up_b; a.down_b = L.down_b;
    a.topk_w = L.topk_w; a.sh_gate = L.sh_gate;
    a.h = (__nv_bfloat16 *)L.h;
    a.ys = L.ys;
    a.status = L.status;
    a.fp4 = nullptr;
    a.stall = L.inject ? L.never : nullptr;
    a.wait_ns = L.wait_ns;
    a.T = T; a.K = L.K; a.E = L.E; a.H = L.H; a.F = L.F; a.Fs = L.Fs; a.Fmax = L.Fmax; a.Tmax = L.Tmax;
    a.act = L.cfg.act;
    a.alpha = L.cfg.act_alpha; a.limit = L.cfg.act_limit;
    a.logits = nullptr; a.rparts = nullptr; a.router_b = nullptr; a.R = L.R; a.router_nt = 1; a.router_S = 1; a.router_bn = 128;
    return a;
}

int launch_experts_tc(const Layer &L, const void *x, int T, int which, cudaStream_t s)
{
    const TensorMaps &m = *L.tmaps;
    TcArgs a = make_tc_args(L, T);
    const int grid = L.num_sms;
    const bool two = tc_lowbit_two_halves(L, T);  // the grouping kernel used the same tiles
    if (which == 1) {
        TcMaps mu{m.xp, m.gate, m.up, m.sh_gate, m.sh_up, m.xp};
        if (L.Fs > 0 && !encode_2d(&mu.sa, x, L.H, (uint64_t)T, TC_BM)) return -1;
        if (L.qfmt == QF_MXFP4) {
            a.fp4 = L.fp4_gu;
            launch_lowbit<EPI_UP, QF_MXFP4>(mu, a, two, grid, s);
        } else if (L.qfmt == QF_Q4) {
            a.fp4 = L.fp4_gu;
            launch_lowbit<EPI_UP, QF_Q4>(mu, a, two, grid, s);
        } else {
            tc_gemm_kernel<EPI_UP, TC_BN_UP, TcMaps><<<grid, TC_THREADS, TcShape<TC_BN_UP>::SMEM, s>>>(mu, a);
        }
    } else {
        TcMaps md{m.h, m.down, m.down, m.sh_down, m.sh_down, m.h};
        if (L.qfmt == QF_MXFP4) {
            a.fp4 = L.fp4_dn;
            launch_lowbit<EPI_DOWN, QF_MXFP4>(md, a, two, grid, s);
        } else if (L.qfmt == QF_Q4) {
            a.fp4 = L.fp4_dn;
            launch_lowbit<EPI_DOWN, QF_Q4>(md, a, two, grid, s);
        } else {
            tc_gemm_kernel<EPI_DOWN, TC_BN_DOWN, TcMaps><<<grid, TC_THREADS, TcShape<TC_BN_DOWN>::SMEM, s>>>(md, a);
        }
    }
    return 1;
}

// K ranges of the router GEMM.  With fewer (token, router-row) tiles than half
// the SMs (few router rows, or few tokens), K is split so that about one tile
// runs per SM, each range at least four 64-wide K blocks, at most
// TC_ROUTER_MAX_SPLITS; the selection kernel then adds the partial sums.
// (Measured on the qwen35moe-, gpt-oss- and mixtral-shaped layers: splits cut
// the router from 25-28 to 15-18 us where it had 16-32 tiles, and cost more
// in the selection kernel than they saved where it had 96 or more.)
int tc_router_splits(const Layer &L, int T)
{
    const int mn = ((T + TC_BM - 1) / TC_BM) * ((L.R + 127) / 128);
    if (2 * mn >= L.num_sms) return 1;  // enough tiles: the partial sums would cost more than they save
    const int S = min((L.num_sms + mn - 1) / mn, min(TC_ROUTER_MAX_SPLITS, (L.H / TC_BK) / 4));
    return max(S, 1);
}

// router logits on the tensor cores: logits[T][R] = x Wr^T (+ b), or with K
// split, partial sums that the selection kernel adds in split order; the x
// tensor map is encoded for this forward's x pointer
int launch_tc_router(const Layer &L, const void *x, int T, cudaStream_t s)
{
    const TensorMaps &m = *L.tmaps;
    TcMaps mr{};
    if (!encode_2d(&mr.a, x, L.H, (uint64_t)T, TC_BM)) return -1;
    mr.b0 = mr.b1 = mr.sb0 = mr.sb1 = m.router;
    TcArgs a = make_tc_args(L, T);
    a.logits = L.logits;
    a.router_b = L.router_b;
    a.R = L.R;
    a.router_nt = (L.R + 127) / 128;
    a.router_S = tc_router_splits(L, T);
    a.router_bn = 128;
    a.rparts = L.router_parts;
    const int tiles = ((T + TC_BM - 1) / TC_BM) * a.router_nt * a.router_S;
    const int grid = tiles < L.num_sms ? tiles : L.num_sms;
    tc_gemm_kernel<EPI_ROUTER, 128, TcMaps><<<grid, TC_THREADS, TcShape<128>::SMEM, s>>>(mr, a);
    return 1;
}

}  // namespace moe
