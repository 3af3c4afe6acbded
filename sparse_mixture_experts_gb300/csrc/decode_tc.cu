// decode_tc.cu -- weight-streaming tensor-core path for small token counts
// (decode batches of up to 16 tokens).
//
// The layer is the same as everywhere ("Qwen3.5-MoE Model Implementation",
// MoE routing; "Phase 19: MoE -- gpt-oss-20b", section 2; "Llama Forward
// Pass", Mixture of Experts):
//   out[t] = sum_j w[t][j] (W_down,e_j act(W_gate,e_j x_t, W_up,e_j x_t) + b_e_j)
//            + sigmoid(w_sh . x_t) W_sh_down (silu(W_sh_gate x_t) * W_sh_up x_t)
// At decode sizes the time is the HBM stream of the selected experts' weights,
// so the tensor cores run with the operands swapped: the weight rows are the
// M = 128 operand, streamed once by TMA through an 8-stage ring, and all (up to
// 16) tokens are the N = 16 operand.
//
//   kernel 1  router logits (one warp per router row); the last block to
//             finish selects the top-k of every token, lists the experts that
//             received tokens ("groups", ascending, then the shared expert) and
//             writes a weight table wtab[g][t] = routing weight of token t for
//             group g (0 when t is not routed to it; sigmoid gate for the
//             shared expert).
//   kernel 2  gate/up: per group, 64 gate rows + 64 up rows x 16 tokens per
//             tile, K = H split into S parts when there are few tiles; the last
//             split to finish sums the partials in split order, applies the
//             activation and stores h'[g][t][f] = wtab[g][t] * act(gate, up).
//   kernel 3  down: per tile of 128 output rows, one TMEM accumulator
//             collects W_down,g h'[g] over all groups (experts in ascending
//             order, then the shared expert), so the routing-weighted sum
//             needs no separate combine; groups split in S parts with the same
//             ordered reduction; the epilogue adds the weighted down biases
//             and writes out.
// Kernels 2 and 3 use programmatic dependent launch so their prologues overlap
// the previous kernel.  All waits are bounded; results are deterministic.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {

constexpr int DT_TOK = 16;                      // N: token columns
constexpr int DT_STAGES = 8;
constexpr int DT_THREADS = 192;
constexpr int DT_A_BYTES = 128 * 64 * 2;        // 16 KB weight tile
constexpr int DT_B_BYTES = DT_TOK * 64 * 2;     // 2 KB token tile
constexpr int DT_STAGE_BYTES = DT_A_BYTES + DT_B_BYTES;
constexpr int DT_ACC = 8;                       // TMEM accumulator buffers (MMA runs ahead of the epilogue)
constexpr int DT_TMEM_COLS = DT_ACC * 16;       // 16 fp32 columns each
constexpr int DT_XCH_BYTES = 64 * DT_TOK * 4;   // up-row values handed to the gate rows
constexpr size_t DT_SMEM = (size_t)DT_STAGES * DT_STAGE_BYTES + 1024 + DT_XCH_BYTES + 512;
constexpr int DT_UNITS_PER_CTA = 16;            // partial-sum slots per CTA

struct DecMaps {
    CUtensorMap gate, up, sh_gate, sh_up;  // box 64 rows x 64
    CUtensorMap down, sh_down;             // box 128 rows x 64
    CUtensorMap x;                         // [T][H], box 16 rows x 64 (encoded per forward)
    CUtensorMap hp;                        // h' [groups*16][Fmax], box 16 rows x 64
};

struct DecArgs {
    const RouteMeta *meta;
    const int *active;
    const float *wtab;      // [groups_max][16]
    const int *topk_idx;
    const float *topk_w;
    const float *gate_b, *up_b, *down_b;
    __nv_bfloat16 *hp;      // [groups_max*16][Fmax]
    float *partials;        // [units][128][16]
    int *tickets;           // [max tiles]
    void *out;
    int *status;
    int T, K, E, H, F, Fs, Fmax;
    int act, out_bf16;
    float alpha, limit;
    int max_units;
};

// ---------------------------------------------------------------------------
// kernel 1: router logits + selection + group tables (T <= 16)
// ---------------------------------------------------------------------------
struct DecRouteArgs {
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *router_w;
    const float *router_b;
    float *logits;
    int *topk_idx;
    float *topk_w;
    float *sh_gate;
    int *counts;
    int *active;
    float *wtab;
    RouteMeta *meta;
    int T, K, E, H, R, Fs;
    int mode, norm;
    float scale;
};

__device__ __forceinline__ bool rt_better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(256) dec_route_kernel(const DecRouteArgs a)
{
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, K = a.K, E = a.E, H = a.H, R = a.R;
    const int r = blockIdx.x * 8 + warp;
    if (r < R) {
        float acc[DT_TOK];
#pragma unroll
        for (int t = 0; t < DT_TOK; ++t) acc[t] = 0.0f;
        const __nv_bfloat16 *w = a.router_w + (size_t)r * H;
#pragma unroll 4
        for (int c = lane; c < H / 8; c += 32) {
            Vec<__nv_bfloat16> wv;
            wv.load_stream(w + (size_t)c * 8);
#pragma unroll
            for (int t = 0; t < DT_TOK; ++t) {
                if (t < T) {
                    Vec<__nv_bfloat16> xv;
                    xv.load(a.x + (size_t)t * H + (size_t)c * 8);
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[t] = fmaf(wv.v[q], xv.v[q], acc[t]);
                }
            }
        }
        const float b = (a.router_b && r < E) ? a.router_b[r] : 0.0f;
#pragma unroll
        for (int t = 0; t < DT_TOK; ++t) {
            if (t < T) {
                float s = warp_sum(acc[t]);
                if (lane == 0) a.logits[(size_t)t * R + r] = s + b;
            }
        }
    }
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&a.meta->ticket, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last block: selection for every token ----
    __shared__ int s_idx[DT_TOK * 32];
    __shared__ float s_w[DT_TOK * 32];
    __shared__ float s_g[DT_TOK];
    __shared__ int s_cnt[1024];
    __shared__ int s_act[1024];
    __shared__ int s_wtot[8];
    __shared__ int s_nact;
    for (int t = warp; t < T; t += 8) {
        const float *l = a.logits + (size_t)t * R;
        float v[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = (lane + 32 * q < E) ? __ldcg(l + lane + 32 * q) : -INFINITY;
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < 32; ++q) mx = fmaxf(mx, v[q]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        unsigned taken = 0;
        int sel_i = -1;
        float sel_v = 0.0f;
        for (int j = 0; j < K; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int e = lane + 32 * q;
                if (e < E && !(taken & (1u << q)) && (bi == 0x7fffffff || rt_better(v[q], e, bv, bi))) {
                    bv = v[q];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi != 0x7fffffff && (bi == 0x7fffffff || rt_better(ov, oi, bv, bi))) { bv = ov; bi = oi; }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) { sel_i = bi; sel_v = bv; }
        }
        float w;
        if (a.mode == MOE_ROUTER_SOFTMAX_TOPK) {
            float z = 0.0f;
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (lane + 32 * q < E) z += __expf(v[q] - mx);
            z = warp_sum(z);
            float p = (lane < K) ? __expf(sel_v - mx) / z : 0.0f;
            float ps = warp_sum(p);
            w = (a.norm ? p / ps : p) * a.scale;
        } else {
            float m0 = __shfl_sync(0xffffffffu, sel_v, 0);
            float ex = (lane < K) ? __expf(sel_v - m0) : 0.0f;
            w = ex / warp_sum(ex);
        }
        if (lane < K) {
            s_idx[t * K + lane] = sel_i;
            s_w[t * K + lane] = w;
        }
        if (lane == 0) s_g[t] = a.Fs > 0 ? 1.0f / (1.0f + __expf(-__ldcg(l + E))) : 0.0f;
    }
    for (int e = threadIdx.x; e < E; e += 256) s_cnt[e] = 0;
    __syncthreads();
    const int P = T * K;
    for (int p = threadIdx.x; p < P; p += 256) atomicAdd(&s_cnt[s_idx[p]], 1);
    __syncthreads();
    {
        int base = 0;
        for (int e0 = 0; e0 < E; e0 += 256) {
            const int e = e0 + threadIdx.x;
            const bool on = e < E && s_cnt[e] > 0;
            const unsigned m = __ballot_sync(0xffffffffu, on);
            if (lane == 0) s_wtot[warp] = __popc(m);
            __syncthreads();
            int before = 0, all = 0;
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) {
                before += w8 < warp ? s_wtot[w8] : 0;
                all += s_wtot[w8];
            }
            if (on) s_act[base + before + __popc(m & ((1u << lane) - 1u))] = e;
            base += all;
            __syncthreads();
        }
        if (threadIdx.x == 0) s_nact = base;
    }
    __syncthreads();
    const int n_act = s_nact;
    for (int p = threadIdx.x; p < P; p += 256) {
        a.topk_idx[p] = s_idx[p];
        a.topk_w[p] = s_w[p];
    }
    for (int e = threadIdx.x; e < E; e += 256) a.counts[e] = s_cnt[e];
    for (int g = threadIdx.x; g < n_act; g += 256) a.active[g] = s_act[g];
    if (a.Fs > 0)
        for (int t = threadIdx.x; t < T; t += 256) a.sh_gate[t] = s_g[t];
    const int n_groups = n_act + (a.Fs > 0 ? 1 : 0);
    for (int q = threadIdx.x; q < n_groups * DT_TOK; q += 256) {
        const int g = q / DT_TOK, t = q - g * DT_TOK;
        float w = 0.0f;
        if (t < T) {
            if (g < n_act) {
                const int e = s_act[g];
                for (int j = 0; j < K; ++j)
                    if (s_idx[t * K + j] == e) w = s_w[t * K + j];
            } else {
                w = s_g[t];
            }
        }
        a.wtab[q] = w;
    }
    if (threadIdx.x == 0) {
        a.meta->n_active = n_act;
        a.meta->n_pairs = P;
        a.meta->ticket = 0;
    }
}

// ---------------------------------------------------------------------------
// schedules (every CTA computes the same ones from the group count)
// ---------------------------------------------------------------------------
// Split count S in [1, smax] minimising the busiest CTA's bytes: ceil(tiles*S /
// G) units of ceil(nkb/S) k-blocks, plus a partial write+read per unit when S >
// 1; at most max_units units.
__device__ __forceinline__ int choose_splits(int tiles, int nkb, int smax, int G, int max_units)
{
    // no split when every CTA already has a tile: a split costs a partial-sum
    // round trip through global memory per unit
    if (tiles >= G) return 1;
    int best = 1;
    long long best_cost = -1;
    for (int S = 1; S <= smax; ++S) {
        if ((long long)tiles * S > max_units && S > 1) break;
        const long long per_cta = ((long long)tiles * S + G - 1) / G;
        const long long cost = per_cta * (((nkb + S - 1) / S) * (long long)DT_STAGE_BYTES + (S > 1 ? 32768 : 0));
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = S; }
    }
    return best;
}

struct UpUnit {
    int g, ft, kb0, kb1, tile, s;
    bool shared;
};

struct UpSched {
    int n_act, groups, tiles_routed, tiles, nkb, S, units;
};

__device__ __forceinline__ UpSched up_sched(const DecArgs &a, int G)
{
    UpSched s;
    s.n_act = a.meta->n_active;
    s.groups = s.n_act + (a.Fs > 0 ? 1 : 0);
    s.tiles_routed = s.n_act * (a.F / 64);
    s.tiles = s.tiles_routed + a.Fs / 64;
    s.nkb = a.H / 64;
    const int smax = max(1, min(16, s.nkb / 2));
    s.S = choose_splits(s.tiles, s.nkb, smax, G, a.max_units);
    s.units = s.tiles * s.S;
    return s;
}

__device__ __forceinline__ UpUnit up_unit(const UpSched &s, int u)
{
    UpUnit x;
    x.tile = u / s.S;
    x.s = u - x.tile * s.S;
    x.kb0 = (int)((long long)s.nkb * x.s / s.S);
    x.kb1 = (int)((long long)s.nkb * (x.s + 1) / s.S);
    if (x.tile < s.tiles_routed) {
        const int per = s.tiles_routed / max(s.n_act, 1);
        x.g = x.tile / per;
        x.ft = x.tile - x.g * per;
        x.shared = false;
    } else {
        x.g = s.n_act;
        x.ft = x.tile - s.tiles_routed;
        x.shared = true;
    }
    return x;
}

struct DownSched {
    int n_act, groups, ot, S, units;
};

__device__ __forceinline__ DownSched down_sched(const DecArgs &a, int G)
{
    DownSched s;
    s.n_act = a.meta->n_active;
    s.groups = s.n_act + (a.Fs > 0 ? 1 : 0);
    s.ot = (a.H + 127) / 128;
    // cost model over group splits: each group is F/64 k-blocks
    const int kb_per_group = a.Fmax / 64;
    s.S = choose_splits(s.ot, s.groups * kb_per_group, s.groups, G, a.max_units);
    // choose_splits counts k-blocks; keep whole groups per split
    s.units = s.ot * s.S;
    return s;
}

// ---------------------------------------------------------------------------
// kernels 2 and 3: weight-streaming tcgen05 GEMMs
// ---------------------------------------------------------------------------
enum { DEC_UP = 0, DEC_DOWN = 1 };

template <int PH>
__global__ void __launch_bounds__(DT_THREADS, 1) dec_tc_kernel(const __grid_constant__ DecMaps maps, const DecArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *xch = reinterpret_cast<float *>(smem + DT_STAGES * DT_STAGE_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + DT_STAGES * DT_STAGE_BYTES + DT_XCH_BYTES);
    uint64_t *empty = full + DT_STAGES;
    uint64_t *acc_full = empty + DT_STAGES;   // [DT_ACC]
    uint64_t *acc_empty = acc_full + DT_ACC;  // [DT_ACC]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + DT_ACC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *bcast = reinterpret_cast<int *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < DT_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < DT_ACC; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 128);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(DT_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (warp == 0 && lane == 0) {
        if (PH == DEC_UP) {
            tmap_prefetch(&maps.gate);
            tmap_prefetch(&maps.up);
            tmap_prefetch(&maps.x);
        } else {
            tmap_prefetch(&maps.down);
            tmap_prefetch(&maps.hp);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // the previous kernel's results (routing tables, h') are read from here on
    pdl_wait();
    pdl_launch_dependents();

    UpSched us;
    DownSched ds;
    int units;
    if (PH == DEC_UP) { us = up_sched(a, G); units = us.units; }
    else { ds = down_sched(a, G); units = ds.units; }

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t last_phase[DT_STAGES];
            bool used[DT_STAGES];
            for (int s = 0; s < DT_STAGES; ++s) used[s] = false, last_phase[s] = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += G) {
                int g0, g1;
                if (PH == DEC_UP) { g0 = 0; g1 = 1; }
                else {
                    const int s = u % ds.S;
                    g0 = (int)((long long)ds.groups * s / ds.S);
                    g1 = (int)((long long)ds.groups * (s + 1) / ds.S);
                }
                for (int gi = g0; gi < g1 && ok; ++gi) {
                    int kb0, kb1;
                    const CUtensorMap *ma, *mb = nullptr;
                    int arow, arow2 = 0, brow;
                    if (PH == DEC_UP) {
                        const UpUnit x = up_unit(us, u);
                        kb0 = x.kb0; kb1 = x.kb1;
                        if (x.shared) { ma = &maps.sh_gate; mb = &maps.sh_up; arow = arow2 = x.ft * 64; }
                        else {
                            const int e = a.active[x.g];
                            ma = &maps.gate; mb = &maps.up;
                            arow = arow2 = e * a.F + x.ft * 64;
                        }
                        brow = 0;
                    } else {
                        const int ot = u / ds.S;
                        const bool shared = gi == ds.n_act;
                        const int fd = shared ? a.Fs : a.F;
                        kb0 = 0; kb1 = fd / 64;
                        if (shared) { ma = &maps.sh_down; arow = ot * 128; }
                        else { ma = &maps.down; arow = a.active[gi] * a.H + ot * 128; }
                        brow = gi * DT_TOK;
                    }
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
                            record_error(a.status, DEV_TIMEOUT_EMPTY_BARRIER);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        uint8_t *sa = smem + stage * DT_STAGE_BYTES;
                        uint8_t *sb = sa + DT_A_BYTES;
                        mbar_arrive_expect_tx(&full[stage], DT_STAGE_BYTES);
                        const int kc = kb * 64;
                        if (PH == DEC_UP) {
                            tma_load_2d(sa, ma, &full[stage], kc, arow);
                            tma_load_2d(sa + DT_A_BYTES / 2, mb, &full[stage], kc, arow2);
                            tma_load_2d(sb, &maps.x, &full[stage], kc, brow);
                        } else {
                            tma_load_2d(sa, ma, &full[stage], kc, arow);
                            tma_load_2d(sb, &maps.hp, &full[stage], kc, brow);
                        }
                        used[stage] = true;
                        last_phase[stage] = phase;
                        if (++stage == DT_STAGES) stage = 0, phase ^= 1;
                    }
                }
            }
            volatile int never = 0;
            for (int s = 0; s < DT_STAGES; ++s)
                if (used[s]) mbar_wait(&full[s], last_phase[s], &never);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, DT_TOK);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            int last_acc = -1;
            uint32_t last_acc_phase = 0;
            for (int u = blockIdx.x; u < units && ok; u += G, ++it) {
                const int b = it % DT_ACC;
                const uint32_t acc_phase = (it / DT_ACC) & 1;
                if (!mbar_wait(&acc_empty[b], acc_phase ^ 1, abort_flag)) {
                    record_error(a.status, DEV_TIMEOUT_ACCUM_FREE);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(b * DT_TOK);
                int nk;
                if (PH == DEC_UP) {
                    const UpUnit x = up_unit(us, u);
                    nk = x.kb1 - x.kb0;
                } else {
                    const int s = u % ds.S;
                    const int g0 = (int)((long long)ds.groups * s / ds.S);
                    const int g1 = (int)((long long)ds.groups * (s + 1) / ds.S);
                    nk = 0;
                    for (int gi = g0; gi < g1; ++gi) nk += (gi == ds.n_act ? a.Fs : a.F) / 64;
                }
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        record_error(a.status, DEV_TIMEOUT_FULL_BARRIER);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * DT_STAGE_BYTES);
                    const uint32_t sb = sa + DT_A_BYTES;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(d_tmem, smem_desc_sw128(sa + k * 32), smem_desc_sw128(sb + k * 32), idesc,
                                 (kb | k) != 0);
                    mma_commit(&empty[stage]);
                    if (++stage == DT_STAGES) stage = 0, phase ^= 1;
                }
                if (!ok) break;
                mma_commit(&acc_full[b]);
                last_acc = b;
                last_acc_phase = acc_phase;
            }
            if (*abort_flag && last_acc >= 0) {
                volatile int never = 0;
                mbar_wait(&acc_full[last_acc], last_acc_phase, &never);
            }
        }
    } else {
        // ------------------------------ epilogue (warps 2..5) ------------------------------
        const int q = warp & 3;
        const int r = q * 32 + lane;                // accumulator row = weight row of the tile
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const int et = threadIdx.x - 64;            // 0..127 within the epilogue group
        int it = 0;
        for (int u = blockIdx.x; u < units; u += G, ++it) {
            const int b = it % DT_ACC;
            const uint32_t acc_phase = (it / DT_ACC) & 1;
            // one thread waits (bounded) and tells the others, so that all 128
            // leave together on a timeout and no named barrier below can hang
            if (et == 0) {
                const bool okw = mbar_wait(&acc_full[b], acc_phase, abort_flag);
                if (!okw) {
                    record_error(a.status, DEV_TIMEOUT_ACCUM_BARRIER);
                    *abort_flag = 1;
                }
                bcast[1] = okw ? 1 : 0;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const bool go = bcast[1] != 0;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (!go) break;
            tc_fence_after();
            uint32_t raw[16];
            tmem_ld16(tmem_base + lane_addr + (uint32_t)(b * DT_TOK), raw);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
            float v[DT_TOK];
#pragma unroll
            for (int t = 0; t < DT_TOK; ++t) v[t] = __uint_as_float(raw[t]);

            int tile, S;
            if (PH == DEC_UP) { const UpUnit x = up_unit(us, u); tile = x.tile; S = us.S; }
            else { tile = u / ds.S; S = ds.S; }

            bool finalize = true;
            if (S > 1) {
                // partial to global, then the last split of the tile reduces in split order
                float4 *dst = reinterpret_cast<float4 *>(a.partials + ((size_t)u * 128 + r) * DT_TOK);
#pragma unroll
                for (int i = 0; i < DT_TOK / 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                __threadfence();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (et == 0) {
                    const int prev = atomicAdd(&a.tickets[(PH == DEC_UP ? 0 : 8192) + tile], 1);
                    const int last = prev == S - 1;
                    if (last) a.tickets[(PH == DEC_UP ? 0 : 8192) + tile] = 0;
                    *bcast = last;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                finalize = *bcast != 0;
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (finalize) {
                    __threadfence();
#pragma unroll
                    for (int t = 0; t < DT_TOK; ++t) v[t] = 0.0f;
                    for (int s = 0; s < S; ++s) {
                        const float4 *src =
                            reinterpret_cast<const float4 *>(a.partials + ((size_t)(tile * S + s) * 128 + r) * DT_TOK);
#pragma unroll
                        for (int i = 0; i < DT_TOK / 4; ++i) {
                            float4 p = __ldcg(src + i);
                            v[4 * i] += p.x; v[4 * i + 1] += p.y; v[4 * i + 2] += p.z; v[4 * i + 3] += p.w;
                        }
                    }
                }
            }
            if (!finalize) continue;

            if (PH == DEC_UP) {
                const UpUnit x = up_unit(us, u);
                // rows 64..127 are the up projections of rows 0..63
                if (r >= 64) {
#pragma unroll
                    for (int t = 0; t < DT_TOK; ++t) xch[(r - 64) * DT_TOK + t] = v[t];
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (r < 64) {
                    const int f = x.ft * 64 + r;
                    const int e = x.shared ? -1 : a.active[x.g];
                    const float bg = (!x.shared && a.gate_b) ? a.gate_b[(size_t)e * a.F + f] : 0.0f;
                    const float bu = (!x.shared && a.up_b) ? a.up_b[(size_t)e * a.F + f] : 0.0f;
                    const float *wt = a.wtab + (size_t)x.g * DT_TOK;
#pragma unroll
                    for (int t = 0; t < DT_TOK; ++t) {
                        const float gv = v[t] + bg, uv = xch[r * DT_TOK + t] + bu;
                        float hval = (x.shared || a.act == MOE_ACT_SWIGLU)
                                         ? activation<MOE_ACT_SWIGLU>(gv, uv, a.alpha, a.limit)
                                         : activation<MOE_ACT_CLAMP_GLU>(gv, uv, a.alpha, a.limit);
                        hval *= __ldcg(wt + t);
                        a.hp[((size_t)x.g * DT_TOK + t) * a.Fmax + f] = __float2bfloat16_rn(hval);
                    }
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
            } else {
                const int row = tile * 128 + r;
                if (row < a.H) {
                    for (int t = 0; t < a.T; ++t) {
                        float o = v[t];
                        if (a.down_b) {
                            for (int j = 0; j < a.K; ++j) {
                                const int p = t * a.K + j;
                                o += __ldcg(a.topk_w + p) * a.down_b[(size_t)__ldcg(a.topk_idx + p) * a.H + row];
                            }
                        }
                        const size_t oi = (size_t)t * a.H + row;
                        if (a.out_bf16) reinterpret_cast<__nv_bfloat16 *>(a.out)[oi] = __float2bfloat16_rn(o);
                        else reinterpret_cast<float *>(a.out)[oi] = o;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(DT_TMEM_COLS));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static bool dec_encode(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool dectc_supported(const Layer &L, int T)
{
    return L.dectc != nullptr && T >= 1 && T <= DT_TOK;
}

int dectc_groups_max(const Layer &L)
{
    const int routed = L.E < DT_TOK * L.K ? L.E : DT_TOK * L.K;
    return routed + (L.Fs > 0 ? 1 : 0);
}

size_t dectc_workspace(const Layer &L, size_t &hp_bytes, size_t &part_bytes, size_t &tab_bytes, size_t &ticket_bytes)
{
    hp_bytes = (size_t)dectc_groups_max(L) * DT_TOK * L.Fmax * 2;
    part_bytes = (size_t)L.num_sms * DT_UNITS_PER_CTA * 128 * DT_TOK * 4;
    tab_bytes = (size_t)dectc_groups_max(L) * DT_TOK * 4;
    ticket_bytes = 16384 * 4;
    return hp_bytes + part_bytes + tab_bytes + ticket_bytes;
}

int dectc_prepare(Layer &L)
{
    DecMaps *m = new (std::nothrow) DecMaps();
    if (!m) return -1;
    bool ok = dec_encode(&m->gate, L.gate_w, L.H, (uint64_t)L.E * L.F, 64) &&
              dec_encode(&m->up, L.up_w, L.H, (uint64_t)L.E * L.F, 64) &&
              dec_encode(&m->down, L.down_w, L.F, (uint64_t)L.E * L.H, 128) &&
              dec_encode(&m->hp, L.dec_hp, L.Fmax, (uint64_t)dectc_groups_max(L) * DT_TOK, DT_TOK);
    if (ok && L.Fs) {
        ok = dec_encode(&m->sh_gate, L.sh_gate_w, L.H, L.Fs, 64) && dec_encode(&m->sh_up, L.sh_up_w, L.H, L.Fs, 64) &&
             dec_encode(&m->sh_down, L.sh_down_w, L.Fs, L.H, 128);
    } else if (ok) {
        m->sh_gate = m->gate;
        m->sh_up = m->up;
        m->sh_down = m->down;
    }
    if (ok)
        ok = cudaFuncSetAttribute(dec_tc_kernel<DEC_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DT_SMEM) ==
                 cudaSuccess &&
             cudaFuncSetAttribute(dec_tc_kernel<DEC_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)DT_SMEM) == cudaSuccess;
    if (!ok) { delete m; return -1; }
    L.dectc = m;
    return 0;
}

void dectc_release(Layer &L)
{
    delete L.dectc;
    L.dectc = nullptr;
}

static DecArgs make_dec_args(const Layer &L, int T, void *out)
{
    DecArgs a;
    a.meta = L.meta;
    a.active = L.active;
    a.wtab = L.dec_wtab;
    a.topk_idx = L.topk_idx;
    a.topk_w = L.topk_w;
    a.gate_b = L.gate_b; a.up_b = L.up_b; a.down_b = L.down_b;
    a.hp = (__nv_bfloat16 *)L.dec_hp;
    a.partials = L.dec_partials;
    a.tickets = L.dec_tickets;
    a.out = out;
    a.status = L.status;
    a.T = T; a.K = L.K; a.E = L.E; a.H = L.H; a.F = L.F; a.Fs = L.Fs; a.Fmax = L.Fmax;
    a.act = L.cfg.act;
    a.out_bf16 = L.cfg.out_dtype == MOE_DT_BF16;
    a.alpha = L.cfg.act_alpha; a.limit = L.cfg.act_limit;
    a.max_units = L.num_sms * DT_UNITS_PER_CTA;
    return a;
}

// which: 0 = router + selection, 1 = gate/up, 2 = down
int launch_dectc(const Layer &L, const void *x, int T, void *out, int which, cudaStream_t s)
{
    if (which == 0) {
        DecRouteArgs r;
        r.x = (const __nv_bfloat16 *)x;
        r.router_w = (const __nv_bfloat16 *)L.router_w;
        r.router_b = L.router_b;
        r.logits = L.logits; r.topk_idx = L.topk_idx; r.topk_w = L.topk_w; r.sh_gate = L.sh_gate;
        r.counts = L.counts; r.active = L.active; r.wtab = L.dec_wtab; r.meta = L.meta;
        r.T = T; r.K = L.K; r.E = L.E; r.H = L.H; r.R = L.R; r.Fs = L.Fs;
        r.mode = L.cfg.router_mode; r.norm = L.cfg.norm_topk_prob; r.scale = L.cfg.weights_scale;
        dec_route_kernel<<<(L.R + 7) / 8, 256, 0, s>>>(r);
        return 1;
    }
    DecMaps m = *L.dectc;
    if (which == 1 && !dec_encode(&m.x, x, L.H, (uint64_t)T, DT_TOK)) return -1;
    DecArgs a = make_dec_args(L, T, out);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(DT_THREADS);
    cfg.dynamicSmemBytes = DT_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = which == 1 ? cudaLaunchKernelEx(&cfg, dec_tc_kernel<DEC_UP>, m, a)
                               : cudaLaunchKernelEx(&cfg, dec_tc_kernel<DEC_DOWN>, m, a);
    return e == cudaSuccess ? 1 : -1;
}

}  // namespace moe
