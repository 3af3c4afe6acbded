// decode_tc.cu -- weight-streaming tensor-core path for small token counts
// (decode batches of up to 16 tokens).
//
// The layer is the same as everywhere ("Qwen3.5-MoE Model Implementation",
// MoE routing; "Phase 19: MoE -- gpt-oss-20b", section 2; "Llama Forward
// Pass", Mixture of Experts):
//   out[t] = sum_j w[t][j] (W_down,e_j act(W_gate,e_j x_t, W_up,e_j x_t) + b_e_j)
//            + sigmoid(w_sh . x_t) W_sh_down (silu(W_sh_gate x_t) * W_sh_up x_t)
// At decode sizes the time is the HBM stream of the selected experts' weights,
// so the tensor cores run with the operands swapped: weight rows are the
// M = 128 operand, streamed once by TMA through an 8-stage ring, and all (up to
// 16) tokens are the N = 16 operand.
//
//   kernel 1  router logits, one CTA per router row (the shared-expert gate
//             vector is row E); it also resets the work counters of kernel 2.
//   kernel 2  one persistent CTA per SM.  Every CTA first selects the top-k of
//             every token from the logits (the same code on the same inputs,
//             so every CTA gets the same routing) and lists the experts that
//             received tokens ("groups", ascending, then the shared expert).
//             Work units, claimed in order from a global counter:
//               gate/up units: 64 gate + 64 up rows of one group x all tokens,
//                 K = H (split in S parts when there are fewer tiles than
//                 CTAs; the last split sums the partials in split order);
//                 epilogue h'[g][t][f] = w(t, g) * act(gate, up), with w(t, g)
//                 the routing weight of token t for group g (0 if not routed,
//                 sigmoid gate for the shared expert); then the group's
//                 completion counter is raised.
//               down units: 128 output rows x all tokens, accumulating
//                 W_down,g h'[g] over a range of groups in one TMEM
//                 accumulator (so the routing-weighted sum needs no combine);
//                 the producer waits for each group's counter before loading
//                 its h' rows; ranges are summed in range order by the last
//                 one to arrive, which adds the weighted down biases and
//                 writes out.
//             All gate/up units are claimed before any down unit, so a waiting
//             down unit only depends on work that CTAs already hold.
// The producer hands each claimed unit to the MMA and epilogue roles through a
// queue (8 slots for bf16 weights, 4 for low-bit ones).  Two MMA threads (four
// for low-bit weights) take the stages of the stream in turn, each into its
// own TMEM accumulator of the unit's slot, and the epilogue adds them.  All
// waits are bounded (about a second); results are deterministic.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "lowbit.cuh"
#include "tc_ptx.cuh"

namespace moe {

constexpr int DT_TOK = 16;                      // N: token columns
constexpr int DT_STAGES = 8;
constexpr int DT_THREADS = 192;                 // producer, MMA, 4 epilogue warps (then the second MMA warp)
constexpr int DT_A_BYTES = 128 * 64 * 2;        // 16 KB weight tile
constexpr int DT_B_BYTES = DT_TOK * 64 * 2;     // 2 KB token tile
constexpr int DT_STAGE_BYTES = DT_A_BYTES + DT_B_BYTES;
constexpr int DT_ACC = 8;                       // unit queue slots (each owns an accumulator per MMA warp)
constexpr int DT_EP_LD = DT_TOK + 1;            // row pitch (floats) of the epilogue's accumulator copy
constexpr int DT_XCH_BYTES = 128 * DT_EP_LD * 4; // the accumulator tile in shared memory
constexpr int DT_MAX_PAIRS = DT_TOK * 32;       // tokens * top_k
// Low-bit weights (MXFP4, Q4): a stage is one 64-wide K block: a token tile
// and one packed block of codes and scales (128 rows x 64 K; see lowbit.cuh).
// The producers' ring holds DT_FP4_RS stages.  DT_FP4_DQG groups of four
// warps take the stages in turn and widen each block to bf16 (MXFP4 exactly,
// by a table lookup per code; Q4 with three bf16 pair FMAs per two codes),
// storing it straight into tensor memory, where the MMA reads its A operand
// (DT_FP4_AS tiles of 32 columns); the token operand is x and h' in bf16 as
// for bf16 weights.  The widened tile never touches shared memory, whose
// bandwidth would otherwise bound the stage rate.
// Measured on the gpt-oss-shaped layer at 16 tokens (per SM, per stage):
// the conversion alone is ALU-bound near 300 cycles, whatever the number of
// groups beyond two; one issuing thread hands the tensor cores an MMA or a
// commit about every 128 cycles (five per stage), so DT_FP4_NM threads issue
// in turn; more A tiles (up to 12) and fewer queue slots changed nothing.
// Three groups beat two and four (four run out of registers).
constexpr int DT_FP4_KPS = 1;                   // K blocks per stage
constexpr int DT_FP4_RS = 24 / DT_FP4_KPS;       // raw stages
constexpr int DT_FP4_DQG = 3;                   // dequantising groups of 4 warps, taking the stages in turn
constexpr int DT_FP4_DQW = 4 * DT_FP4_DQG;      // dequantising warps
constexpr int DT_FP4_NP = 4;                    // producer threads
constexpr int DT_BF16_NP = 1;                   // producer threads, bf16 weights
constexpr int DT_FP4_NM = 4;                    // MMA issuing threads
constexpr int DT_FP4_ACC = 4;                   // unit queue slots
constexpr int DT_FP4_TMEM_COLS = 512;
constexpr int DT_FP4_A_COL = DT_FP4_ACC * DT_FP4_NM * DT_TOK;  // first A-tile column, after the accumulators
constexpr int DT_FP4_AS = (DT_FP4_TMEM_COLS - DT_FP4_A_COL) / (32 * DT_FP4_KPS);  // A tiles in tensor memory

// QF: the routed experts' format -- 0 bf16 (TMA tiles), 1 MXFP4, 2 Q4 (packed
// low-bit blocks, widened to bf16 in tensor memory)
template <int QF>
struct DtShape {
    static constexpr bool FP4 = QF != 0;  // packed low-bit weights (either format)
    static constexpr int BLK = QF == 2 ? LOWBIT_BLK_Q4 : LOWBIT_BLK_MXFP4;  // bytes of a packed block
    // bf16: producer, MMA, 4 epilogue warps, a second MMA warp; low-bit: producer, MMA, 4 epilogue
    // warps, DQW dequantising warps, a second MMA warp, a warp of three more producer threads and
    // NM - 2 more MMA warps
    static constexpr int NM = FP4 ? DT_FP4_NM : 2;                  // MMA warps (one issuing thread each)
    static constexpr int NP = FP4 ? DT_FP4_NP : DT_BF16_NP;         // producer threads
    // the warp of producer threads 1 .. NP - 1
    static constexpr int PROD2_WARP = FP4 ? 7 + DT_FP4_DQW : 7;
    static constexpr int THREADS = FP4 ? DT_THREADS + 32 * (DT_FP4_DQW + 2 + NM - 2)
                                       : DT_THREADS + 32 + (NP > 1 ? 32 : 0);
    static constexpr int ACC = FP4 ? DT_FP4_ACC : DT_ACC;           // unit queue slots
    // the MMA warps in issuing order: warp 1, then 6 (bf16) or 6 + DQW, 8 + DQW, 9 + DQW (low-bit)
    static __device__ __forceinline__ int mma_index(int warp)
    {
        if (warp == 1) return 0;
        if (warp == (FP4 ? 6 + DT_FP4_DQW : 6)) return 1;
        if (FP4 && warp >= 8 + DT_FP4_DQW && warp < 6 + DT_FP4_DQW + NM) return warp - 6 - DT_FP4_DQW;
        return -1;
    }
    static constexpr int RS = FP4 ? DT_FP4_RS : DT_STAGES;   // producer ring
    static constexpr int TMEM_COLS = FP4 ? DT_FP4_TMEM_COLS : ACC * NM * DT_TOK;
    static constexpr int KPS = FP4 ? DT_FP4_KPS : 1;        // K blocks per stage
    // smem: bf16 [RS][A | B]; MXFP4 [RS][KPS][B] [RS][KPS][block]
    static constexpr int B_OFF = FP4 ? 0 : DT_A_BYTES;      // first B tile
    static constexpr int B_STRIDE = FP4 ? KPS * DT_B_BYTES : DT_STAGE_BYTES;
    static constexpr int A_STRIDE = DT_STAGE_BYTES;         // bf16 only
    static constexpr int BLK_OFF = RS * KPS * DT_B_BYTES;   // MXFP4 only
    static constexpr int BLK_STRIDE = KPS * BLK;
    static constexpr int RING = FP4 ? (BLK_OFF + RS * BLK_STRIDE + 1023) / 1024 * 1024 : DT_STAGES * DT_STAGE_BYTES;
    static constexpr int TAB_BYTES = QF == 1 ? 256 * (int)sizeof(Fp4Table) : 0;  // MXFP4 -> bf16 tables, one per scale byte
    static constexpr size_t SMEM = (size_t)RING + 1024 + DT_XCH_BYTES + 1024 + TAB_BYTES;
};
static_assert(DT_FP4_KPS == 1, "one K block per low-bit stage (two per stage faulted in a timing variant)");
static_assert(DtShape<1>::ACC * DtShape<1>::NM * DT_TOK <= DT_FP4_A_COL &&
                  DT_FP4_A_COL + DT_FP4_AS * DT_FP4_KPS * 32 <= DT_FP4_TMEM_COLS,
              "low-bit accumulators and A tiles fit the tensor memory allocation");
static_assert(DtShape<0>::TMEM_COLS <= 512 && DtShape<0>::ACC * DtShape<0>::NM <= 16 && DtShape<1>::NM <= 4 &&
                  DT_FP4_AS >= 4 && DT_FP4_AS <= 16 && DT_FP4_ACC <= DT_ACC,
              "accumulators fit; the drain, queue and tile barriers fit their shared-memory slots");
static_assert(DT_FP4_RS <= 32 && DT_STAGES <= 32, "the producer's per-stage masks are 32 bits");
static_assert(DtShape<1>::SMEM + 13 * 1024 <= 227 * 1024, "MXFP4 ring, tables and static shared memory fit a CTA");
static_assert(DtShape<2>::SMEM + 13 * 1024 <= 227 * 1024, "Q4 ring and static shared memory fit a CTA");
constexpr int DT_UNITS_PER_CTA = 16;            // partial-sum slots per CTA
constexpr int DT_SATURATING_CTAS = 128;         // CTAs streaming at once that saturate HBM
constexpr int DT_UP_MIN_KB = 8;                 // smallest gate/up split, in 64-wide K blocks
constexpr int DT_DOWN_GUIDE = 1;                // down ranges: a round of units takes 1/GUIDE of the K blocks left
constexpr int DT_DOWN_MIN_KB = 8;               // smallest down range, in 64-wide K blocks (but the last)
constexpr int DT_MAX_DOWN_SPLITS = 64;
constexpr int DT_CLAIM_AHEAD = 4;               // stages before a unit's end at which the next one is claimed
constexpr int DT_TICKET_DOWN = 8192;            // offset of the down tiles' tickets
constexpr int DT_GROUP_DONE = 12288;            // offset of the per-group completion counters
constexpr int DT_DONE_STRIDE = 32;              // one 128-byte line per group counter
constexpr int DT_NEXT_UNIT = 32736;             // offset of the work counter (a line of its own)
constexpr int DT_COUNTERS = 32768;              // ints

struct DecMaps {
    CUtensorMap gate, up, sh_gate, sh_up;  // box 64 rows x 64
    CUtensorMap down, sh_down;             // box 128 rows x 64
    CUtensorMap x;                         // [T][H], box 16 rows x 64 (encoded per forward)
    CUtensorMap hp;                        // h' [groups*16][Fmax], box 16 rows x 64
};

struct DecArgs {
    const float *logits;  // [T][R]
    int *topk_idx;        // outputs for moe_get_routing & co. (written by CTA 0)
    float *topk_w;
    float *sh_gate;
    int *counts;
    int *active;
    RouteMeta *meta;
    const float *gate_b, *up_b, *down_b;
    void *hp;             // [groups_max*16][Fmax], bf16
    const uint8_t *gu_fp4, *dn_fp4;  // MXFP4 weights, packed blocks (see Layer)
    int ot;               // down output tiles of 128 rows
    float *partials;      // [gate/up, down][units][T][128]
    int *counters;        // tickets, group completion, work counter
    void *out;
    int *status;
    int T, K, E, H, F, Fs, Fmax, R;
    int mode, norm;
    float scale;
    int act, out_bf16;
    float alpha, limit;
    int max_units;
    unsigned long long wait_ns;  // bound of a wait on another CTA's activations
    int inject;                  // test-only: dependency waits that never complete
    const int *slot_of;          // expert residency: [E] the slot holding each expert's weights (else NULL)
    int accumulate;              // a later chunk of a forward: the expert counts add up
};

// ---------------------------------------------------------------------------
// kernel 1: router logits (T <= 16), one CTA per router row
// ---------------------------------------------------------------------------
struct DecRouteArgs {
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *router_w;
    const float *router_b;
    float *logits;
    int *counters;
    int T, E, H, R;
    int n_reset;  // per-group counters to clear
};

__global__ void __launch_bounds__(256) dec_route_kernel(const DecRouteArgs a)
{
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, H = a.H, R = a.R;
    if (blockIdx.x == 0) {
        // kernel 2 of the previous forward has finished (stream order)
        for (int i = threadIdx.x; i < a.n_reset; i += 256) a.counters[DT_GROUP_DONE + i * DT_DONE_STRIDE] = 0;
        if (threadIdx.x == 0) a.counters[DT_NEXT_UNIT] = 0;
    }
    __shared__ float s_part[8][DT_TOK];
    const int r = blockIdx.x;
    float acc[DT_TOK];
#pragma unroll
    for (int t = 0; t < DT_TOK; ++t) acc[t] = 0.0f;
    const __nv_bfloat16 *w = a.router_w + (size_t)r * H;
    for (int c = threadIdx.x; c < H / 8; c += 256) {
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
#pragma unroll
    for (int t = 0; t < DT_TOK; ++t) {
        if (t < T) {
            const float sum = warp_sum(acc[t]);
            if (lane == 0) s_part[warp][t] = sum;
        }
    }
    __syncthreads();
    if (threadIdx.x < T) {
        float sum = 0.0f;
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) sum += s_part[w8][threadIdx.x];
        const float b = (a.router_b && r < a.E) ? a.router_b[r] : 0.0f;
        a.logits[(size_t)threadIdx.x * R + r] = sum + b;
    }
}

// ---------------------------------------------------------------------------
// schedules (every CTA computes the same ones from the group count)
// ---------------------------------------------------------------------------
// Gate/up splits.  One SM streams at most about 120 GB/s by TMA alone and
// less beside the MMA and handoffs, so about 128 CTAs streaming at once
// saturate HBM.  Below that many tiles every tile is split along K into S
// parts.  Otherwise the tiles of the last, partial round of claims (tiles mod
// G, when that is at most G / 2) are split so that round has about G units of
// at least DT_UP_MIN_KB K blocks, and the others are not.  Each split costs a partial-sum round trip
// through L2.  Sets the first split tile and the split count of the rest.
__device__ __forceinline__ void up_splits(int tiles, int nkb, int G, int max_units, int &full, int &S)
{
    const int smax = max(1, min(16, nkb / DT_UP_MIN_KB));
    int r;
    if (tiles < DT_SATURATING_CTAS) {
        full = 0;
        r = tiles;
        S = min(smax, (DT_SATURATING_CTAS + tiles - 1) / tiles);
    } else {
        r = tiles % G;
        if (2 * r > G) r = 0;  // the last round is more than half full already
        full = tiles - r;
        S = r > 0 ? min(smax, (G + r - 1) / r) : 1;
    }
    while (S > 1 && r * S > max_units) --S;
    S = max(1, S);
}

// Down split boundaries, the same in every CTA.  The down projection's K is
// the concatenation of every group's h' (F / 64 blocks per routed expert, then
// Fs / 64 for the shared expert); a down unit is one output tile over a range
// of those K blocks, which may span groups.  Units are claimed split-major, so
// the ranges shrink toward the end (guided self-scheduling): about one round
// of units (G / ot splits) covers 1 / DT_DOWN_GUIDE of the blocks still left,
// down to DT_DOWN_MIN_KB; at most maxs splits.  Returns the split count;
// b[0..S] are the boundaries in K blocks.
__device__ __forceinline__ int down_bounds(int total_kb, int ot, int G, int maxs, int *b)
{
    const int per_round = max(1, G / ot) * DT_DOWN_GUIDE;
    int s = 0, k = 0;
    b[0] = 0;
    while (k < total_kb) {
        const int left = total_kb - k;
        int size = max(DT_DOWN_MIN_KB, (left + per_round - 1) / per_round);
        if (s == maxs - 1 || size > left) size = left;
        k += size;
        b[++s] = k;
    }
    return s;
}

struct Sched {
    int n_act, groups;
    int tiles_routed, up_tiles, nkb, up_full, S_up, up_units;  // gate/up: tiles [up_full, up_tiles) are split S_up ways
    int ot;                                          // down output tiles (the split count comes later)
    int per, kb_routed, total_kb;                    // down K blocks: per routed group, all routed, all
};

__device__ __forceinline__ Sched make_sched(const DecArgs &a, int n_act, int G)
{
    Sched s;
    s.n_act = n_act;
    s.groups = n_act + (a.Fs > 0 ? 1 : 0);
    s.tiles_routed = n_act * (a.F / 64);
    s.up_tiles = s.tiles_routed + a.Fs / 64;
    s.nkb = a.H / 64;
    up_splits(s.up_tiles, s.nkb, G, a.max_units, s.up_full, s.S_up);
    s.up_units = s.up_full + (s.up_tiles - s.up_full) * s.S_up;
    s.ot = (a.H + 127) / 128;
    s.per = a.F / 64;
    s.kb_routed = n_act * s.per;
    s.total_kb = s.kb_routed + a.Fs / 64;
    return s;
}

// gate/up unit u (< up_units): tiles in group-major order, the split ones last;
// split s of S, whose partial goes to slot pslot + s
struct UpUnit {
    int g, ft, kb0, kb1, tile, s, S, pslot;
    bool shared;
};

__device__ __forceinline__ UpUnit up_unit(const Sched &s, int u, int F)
{
    UpUnit x;
    if (u < s.up_full) {
        x.tile = u;
        x.s = 0;
        x.S = 1;
        x.pslot = 0;
    } else {
        const int v = u - s.up_full;
        const int i = v / s.S_up;
        x.tile = s.up_full + i;
        x.s = v - i * s.S_up;
        x.S = s.S_up;
        x.pslot = i * s.S_up;
    }
    x.kb0 = s.nkb * x.s / x.S;
    x.kb1 = s.nkb * (x.s + 1) / x.S;
    const int per = F / 64;
    if (x.tile < s.tiles_routed) {
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

// down unit d (= u - up_units): split s = d / ot (so early units need early
// groups), output tile d % ot, K blocks [kb0, kb1) of the concatenated groups
struct DnUnit {
    int tile, s, kb0, kb1;
};

__device__ __forceinline__ DnUnit dn_unit(const Sched &s, int d, const int *bounds)
{
    DnUnit x;
    x.s = d / s.ot;
    x.tile = d - x.s * s.ot;
    x.kb0 = bounds[x.s];
    x.kb1 = bounds[x.s + 1];
    return x;
}

// the group of concatenated down K block kb, and the block within that group
__device__ __forceinline__ int dn_group(const Sched &s, int kb, int &local)
{
    if (kb < s.kb_routed) {
        const int g = kb / s.per;
        local = kb - g * s.per;
        return g;
    }
    local = kb - s.kb_routed;
    return s.n_act;
}

// v[t] += the S split partials of row r, in split order; U splits' loads are
// in flight at a time (TT >= T token slots)
template <int TT, int U>
__device__ __forceinline__ void sum_partials(const float *pt, int S, int T, int r, float (&v)[DT_TOK])
{
    for (int s0 = 0; s0 < S; s0 += U) {
        float pv[U][TT];
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int t = 0; t < TT; ++t)
                pv[j][t] = (s0 + j < S && t < T) ? __ldcg(pt + ((size_t)(s0 + j) * T + t) * 128 + r) : 0.0f;
#pragma unroll
        for (int j = 0; j < U; ++j)
#pragma unroll
            for (int t = 0; t < TT; ++t) v[t] += pv[j][t];
    }
}

// routing weight of token t for group g (0 when t is not routed to it)
__device__ __forceinline__ float group_weight(int g, int t, int n_act, int K, const int *s_act, const int *s_idx,
                                              const float *s_w, const float *s_gsh)
{
    if (g == n_act) return s_gsh[t];
    const int e = s_act[g];
    float w = 0.0f;
    for (int j = 0; j < K; ++j)
        if (s_idx[t * K + j] == e) w = s_w[t * K + j];
    return w;
}

// ---------------------------------------------------------------------------
// kernel 2: selection + gate/up + down, persistent, dynamic work claiming
// ---------------------------------------------------------------------------
template <int QF>
__global__ void __launch_bounds__(DtShape<QF>::THREADS, 1) dec_experts_kernel(const __grid_constant__ DecMaps maps,
                                                                               const DecArgs a)
{
    using Sh = DtShape<QF>;
    constexpr bool FP4 = Sh::FP4;  // packed low-bit weights
    constexpr int THREADS = Sh::THREADS;
    constexpr int RS = Sh::RS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *xch = reinterpret_cast<float *>(smem + Sh::RING);
    Fp4Table *fp4tab = reinterpret_cast<Fp4Table *>(smem + Sh::RING + DT_XCH_BYTES + 1024);  // MXFP4 only
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Sh::RING + DT_XCH_BYTES);  // [RS] raw stage landed
    uint64_t *empty = full + RS;              // [RS] raw stage consumed
    constexpr int ACC = Sh::ACC;
    uint64_t *acc_full = empty + RS;          // [ACC]
    uint64_t *uq_full = acc_full + ACC;       // [ACC] unit handed out
    uint64_t *uq_empty = uq_full + ACC;       // [ACC] unit finished, slot and accumulator free
    uint64_t *deq = uq_empty + ACC;           // [DT_FP4_AS] low-bit: the A tile is in tensor memory
    uint64_t *drain = deq + DT_FP4_AS;        // [NM] an MMA thread's own completion, after an abort
    int *uq = reinterpret_cast<int *>(drain + Sh::NM);  // [ACC]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(uq + ACC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *bcast = reinterpret_cast<int *>(tmem_slot + 2);  // [4]

    __shared__ int s_idx[DT_MAX_PAIRS];
    __shared__ float s_w[DT_MAX_PAIRS];
    __shared__ float s_gsh[DT_TOK];
    __shared__ int s_cnt[1024];
    __shared__ uint32_t s_mask[32];  // bit e: expert e has at least one pair
    __shared__ int s_act[DT_MAX_PAIRS];
    __shared__ int s_wslot[DT_MAX_PAIRS];  // where each active expert's weights are: s_act, or its slot
    __shared__ int s_dnb[DT_MAX_DOWN_SPLITS + 1];  // down split boundaries
    __shared__ int s_sdn;                          // down split count
    __shared__ __align__(8) uint64_t s_bnd_bar;    // s_dnb and s_sdn are written
    __shared__ float s_wt[DT_TOK];  // routing weight per token of the current gate/up unit

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int T = a.T, K = a.K, E = a.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&s_bnd_bar, 1);
        for (int b = 0; b < ACC; ++b) {
            mbar_init(&acc_full[b], Sh::NM);
            mbar_init(&uq_full[b], 1);
            mbar_init(&uq_empty[b], Sh::NP);  // the epilogue and the following producers
        }
        if (FP4)
            for (int s = 0; s < DT_FP4_AS; ++s) mbar_init(&deq[s], DT_FP4_DQW / DT_FP4_DQG);
        for (int m = 0; m < Sh::NM; ++m) mbar_init(&drain[m], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(Sh::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (warp == 0 && lane == 0) {
        tmap_prefetch(&maps.gate);
        tmap_prefetch(&maps.up);
        tmap_prefetch(&maps.x);
        tmap_prefetch(&maps.down);
        tmap_prefetch(&maps.hp);
    }
    for (int e = threadIdx.x; e < E; e += THREADS) s_cnt[e] = 0;
    if (threadIdx.x < 32) s_mask[threadIdx.x] = 0u;
    if constexpr (QF == 1)
        for (int i = threadIdx.x; i < 256; i += THREADS) fp4tab[i] = mxfp4_table((uint32_t)i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // the selection's parameters are read before the wait, so that their
    // first (cold) reads overlap it
    asm volatile("" ::"l"(a.logits), "r"(a.R), "r"(a.Fs), "r"(a.mode), "r"(a.norm), "f"(a.scale), "l"(a.counters));

    // the router's logits (and the reset counters) are read from here on
    pdl_wait();
    // the producer's first claim; its latency overlaps the selection below
    int first_unit = 0;
    if (threadIdx.x == 0) first_unit = atomicAdd(a.counters + DT_NEXT_UNIT, 1);

    // ---- routing, the same in every CTA ----
    // two tokens per warp at a time, so their load latencies and dependent
    // reductions overlap
    constexpr int NW = THREADS / 32;
    for (int t = warp; t < T; t += 2 * NW) {
        const int t2 = t + NW;
        const bool two = t2 < T;
        const float *l = a.logits + (size_t)t * a.R;
        const float *l2 = a.logits + (size_t)(two ? t2 : t) * a.R;
        // the shared expert's gate logit sits after the E router logits
        const float gl = (lane == 0 && a.Fs > 0) ? __ldcg(l + E) : 0.0f;
        const float gl2 = (lane == 0 && a.Fs > 0 && two) ? __ldcg(l2 + E) : 0.0f;
        int sel_i[2];
        float sel_v[2], w[2];
        warp_select2_any(l, l2, E, K, a.mode, a.norm, a.scale, lane, sel_i, sel_v, w);
        if (lane < K) {
            s_idx[t * K + lane] = sel_i[0];
            s_w[t * K + lane] = w[0];
            atomicAdd(&s_cnt[sel_i[0]], 1);
            atomicOr(&s_mask[sel_i[0] >> 5], 1u << (sel_i[0] & 31));
            if (two) {
                s_idx[t2 * K + lane] = sel_i[1];
                s_w[t2 * K + lane] = w[1];
                atomicAdd(&s_cnt[sel_i[1]], 1);
                atomicOr(&s_mask[sel_i[1] >> 5], 1u << (sel_i[1] & 31));
            }
        }
        if (lane == 0) {
            s_gsh[t] = a.Fs > 0 ? 1.0f / (1.0f + __expf(-gl)) : 0.0f;
            if (two) s_gsh[t2] = a.Fs > 0 ? 1.0f / (1.0f + __expf(-gl2)) : 0.0f;
        }
    }
    __syncthreads();
    const int P = T * K;
    // active experts in ascending order: each one's slot is the number of
    // selected experts below it
    const int nwords = (E + 31) / 32;
    int n_act = 0;
    for (int wd = 0; wd < nwords; ++wd) n_act += __popc(s_mask[wd]);
    for (int e = threadIdx.x; e < E; e += THREADS) {
        const uint32_t m = s_mask[e >> 5];
        if ((m >> (e & 31)) & 1u) {
            int r = __popc(m & ((1u << (e & 31)) - 1u));
            for (int wd = 0; wd < (e >> 5); ++wd) r += __popc(s_mask[wd]);
            s_act[r] = e;
            int w = e;
            if (a.slot_of) {
                w = a.slot_of[e];
                if (w < 0) {  // not resident: an inconsistent table; slot 0 keeps the reads in bounds
                    record_error(a.status, DEV_NOT_RESIDENT);
                    w = 0;
                }
            }
            s_wslot[r] = w;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int p = threadIdx.x; p < P; p += THREADS) {
            a.topk_idx[p] = s_idx[p];
            a.topk_w[p] = s_w[p];
        }
        for (int e = threadIdx.x; e < E; e += THREADS) a.counts[e] = (a.accumulate ? a.counts[e] : 0) + s_cnt[e];
        for (int g = threadIdx.x; g < n_act; g += THREADS) a.active[g] = s_act[g];
        if (a.Fs > 0)
            for (int t = threadIdx.x; t < T; t += THREADS) a.sh_gate[t] = s_gsh[t];
        if (threadIdx.x == 0) {
            a.meta->n_active = n_act;
            a.meta->n_pairs = P;
        }
    }
    const Sched sc = make_sched(a, n_act, G);
    int *tickets = a.counters;
    int *group_done = a.counters + DT_GROUP_DONE;
    int *next_unit = a.counters + DT_NEXT_UNIT;

    if (warp == 0 || (Sh::NP > 1 && warp == Sh::PROD2_WARP)) {
        // ------------------------------ producer(s) ------------------------------
        // Producer 0 claims the units and hands them out.  NP - 1 more
        // producer threads follow the queue, and producer p issues the stages
        // whose index in the stream is p mod NP, since one thread hands the
        // copy engine a copy only every few hundred cycles.
        constexpr int NP = Sh::NP;
        const int pw = warp == 0 ? (lane == 0 ? 0 : NP) : (lane < NP - 1 ? 1 + lane : NP);
        if (pw < NP) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t used = 0, last_phase = 0;  // per stage: loads issued, parity of the last
            uint32_t gs = 0;                    // index of the next stage in the stream
            int qi = 0;
            uint32_t qph = 0;
            bool ok = true;
            int u_next = first_unit;
            bool bounds = false;
            while (ok) {
                int u;
                if (pw == 0) {
                    u = u_next;
                    if (u >= sc.up_units) {
                        // the down split count is computed off the critical path (epilogue role)
                        if (!bounds && !mbar_wait(&s_bnd_bar, 0, abort_flag)) {
                            record_error(a.status, DEV_TIMEOUT_ACCUM_BARRIER);
                            *abort_flag = 1;
                            u = -1;
                        }
                        bounds = true;
                        if (u >= sc.up_units + sc.ot * s_sdn) u = -1;
                    }
                    if (!mbar_wait(&uq_empty[qi], qph ^ 1, abort_flag)) {
                        record_error(a.status, DEV_TIMEOUT_ACCUM_FREE);
                        *abort_flag = 1;
                        break;
                    }
                    uq[qi] = u;
                    mbar_arrive(&uq_full[qi]);
                } else {
                    if (!mbar_wait(&uq_full[qi], qph, abort_flag)) {
                        record_error(a.status, DEV_TIMEOUT_ACCUM_FREE);
                        *abort_flag = 1;
                        break;
                    }
                    u = uq[qi];
                    // the slot may be handed out again only once this thread has read it
                    mbar_arrive(&uq_empty[qi]);
                }
                if (++qi == ACC) qi = 0, qph ^= 1;
                if (u < 0) break;
                const bool is_up = u < sc.up_units;
                UpUnit ux;
                DnUnit dn;
                int seg_k, seg_end;  // K blocks of the unit (down: of the concatenated groups)
                if (is_up) {
                    ux = up_unit(sc, u, a.F);
                    seg_k = ux.kb0;
                    seg_end = ux.kb1;
                } else {
                    dn = dn_unit(sc, u - sc.up_units, s_dnb);
                    seg_k = dn.kb0;
                    seg_end = dn.kb1;
                }
                int left = seg_end - seg_k;
                const int unit_nk = left;
                int pos = 0;          // K block of the unit
                bool merged = false;  // MXFP4: this stage's second block came with the first
                // the next unit is claimed a few stages before this one ends, so
                // the counter's round trip overlaps this unit's loads.  Claims stay
                // in order: a CTA holds at most one unclaimed-ahead unit, and a
                // down unit only waits for gate/up units, which never wait.
                bool claimed = pw != 0;  // only producer 0 claims
                // one segment per group the unit's K blocks fall in (gate/up: one)
                while (seg_k < seg_end && ok) {
                    int kb0, kb1, arow, brow, wexp;  // wexp: the segment's expert (MXFP4 weights)
                    const CUtensorMap *ma, *mb = nullptr;
                    if (is_up) {
                        kb0 = seg_k; kb1 = seg_end;
                        seg_k = seg_end;
                        wexp = ux.shared ? 0 : s_wslot[ux.g];
                        if (ux.shared) { ma = &maps.sh_gate; mb = &maps.sh_up; arow = ux.ft * 64; }
                        else { ma = &maps.gate; mb = &maps.up; arow = s_wslot[ux.g] * a.F + ux.ft * 64; }
                        brow = 0;
                    } else {
                        int local;
                        const int gi = dn_group(sc, seg_k, local);
                        const bool shared = gi == sc.n_act;
                        const int fd = shared ? a.Fs : a.F;
                        const int n = min(fd / 64 - local, seg_end - seg_k);
                        kb0 = local; kb1 = local + n;
                        seg_k += n;
                        wexp = shared ? 0 : s_wslot[gi];
                        if (shared) { ma = &maps.sh_down; arow = dn.tile * 128; }
                        else { ma = &maps.down; arow = s_wslot[gi] * a.H + dn.tile * 128; }
                        brow = gi * DT_TOK;
                        // h'[gi] is complete once every gate/up tile of the group is
                        // (only waited for by a producer with a stage in the segment:
                        // its stages are those of stream index gs .. gs + ns - 1)
                        const int need = fd / 64 + a.inject;  // (never reached under fault injection)
                        int *done = group_done + gi * DT_DONE_STRIDE;
                        const int ns = (pos % Sh::KPS + n + Sh::KPS - 1) / Sh::KPS;
                        if ((ns >= NP || (int)(((uint32_t)pw + NP - gs % NP) % NP) < ns) && ld_acquire(done) < need) {
                            // poll with a short back-off: many producers may wait on
                            // the same counter, and the increment must get through
                            const unsigned long long t0 = globaltimer();
                            while (ld_acquire(done) < need) {
                                __nanosleep(128);
                                if (*abort_flag || globaltimer() - t0 > a.wait_ns) {
                                    record_error(a.status, DEV_TIMEOUT_DEPENDENCY);
                                    *abort_flag = 1;
                                    ok = false;
                                    break;
                                }
                            }
                        }
                        fence_proxy_async_global();
                        if (!ok) break;
                    }
                    for (int kb = kb0; kb < kb1; ++kb, --left, ++pos) {
                        if (!claimed && left <= DT_CLAIM_AHEAD) {
                            u_next = atomicAdd(next_unit, 1);
                            claimed = true;
                        }
                        const int sub = pos % Sh::KPS;  // K block within the stage
                        if ((int)(gs % NP) == pw) {
                            if (sub == 0) {
                                if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
                                    record_error(a.status, DEV_TIMEOUT_EMPTY_BARRIER);
                                    *abort_flag = 1;
                                    ok = false;
                                    break;
                                }
                                // the one arrival of the stage's full barrier, with every byte its
                                // copies below complete (bf16: A and the token tile; MXFP4: per K
                                // block a packed block and a token tile)
                                const int nkb = min(Sh::KPS, unit_nk - pos);
                                mbar_arrive_expect_tx(&full[stage], FP4 ? nkb * (DT_B_BYTES + Sh::BLK) : DT_STAGE_BYTES);
                            }
                            uint8_t *sa = smem + stage * Sh::A_STRIDE;  // bf16 only
                            uint8_t *sb = smem + Sh::B_OFF + stage * Sh::B_STRIDE + sub * DT_B_BYTES;
                            const int kc = kb * 64;
                            if (FP4) {
                                // the packed block(s) of this (row block, K block): one copy for
                                // both blocks of a stage when they are adjacent (the same segment);
                                // the token tile by TMA
                                const size_t blk = is_up ? ((size_t)wexp * (a.F / 64) + ux.ft) * (a.H / 64) + kb
                                                         : ((size_t)wexp * a.ot + dn.tile) * (a.F / 64) + kb;
                                if (sub == 0 || !merged) {
                                    merged = sub == 0 && Sh::KPS == 2 && kb + 1 < kb1;  // (KPS <= 2)
                                    const uint32_t nb = merged ? 2 : 1;
                                    bulk_load(smem + Sh::BLK_OFF + stage * Sh::BLK_STRIDE + sub * Sh::BLK,
                                              (is_up ? a.gu_fp4 : a.dn_fp4) + blk * Sh::BLK, nb * Sh::BLK,
                                              &full[stage]);
                                }
                                tma_load_2d(sb, is_up ? &maps.x : &maps.hp, &full[stage], kc, brow);
                            } else if (is_up) {
                                tma_load_2d(sa, ma, &full[stage], kc, arow);
                                tma_load_2d(sa + DT_A_BYTES / 2, mb, &full[stage], kc, arow);
                                tma_load_2d(sb, &maps.x, &full[stage], kc, brow);
                            } else {
                                tma_load_2d(sa, ma, &full[stage], kc, arow);
                                tma_load_2d(sb, &maps.hp, &full[stage], kc, brow);
                            }
                            used |= 1u << stage;
                            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                        }
                        if (sub == Sh::KPS - 1 || pos == unit_nk - 1) {  // the stage is complete
                            if (++stage == RS) stage = 0, phase ^= 1;
                            ++gs;
                        }
                    }
                }
                if (!claimed) u_next = atomicAdd(next_unit, 1);
            }
            if (pw == 0 && *abort_flag) {
                // let the other roles leave: hand out the end-of-work marker
                for (int i = 0; i < ACC; ++i) {
                    uq[qi] = -1;
                    mbar_arrive(&uq_full[qi]);
                    if (++qi == ACC) qi = 0, qph ^= 1;
                }
            }
            volatile int never = 0;
            for (int s = 0; s < RS; ++s)
                if ((used >> s) & 1u) mbar_wait(&full[s], (last_phase >> s) & 1u, &never);
        }
    } else if (Sh::mma_index(warp) >= 0) {
        // ------------------------------ MMA issuers ------------------------------
        // NM threads, each in a warp of its own, take the stages in turn (by
        // their index in the stream) into accumulators of their own, which the
        // epilogue adds.  An issuing thread can hand the tensor cores about one
        // MMA (or commit) per 128 cycles, whatever N is, while the tensor cores
        // take them from several threads at once; so at N = 16 one thread's
        // issue rate would bound the stream (two for bf16 weights, four for the
        // smaller low-bit stages).  Low-bit weights: A is the tile the
        // dequantising warps left in tensor memory.
        constexpr int NM = Sh::NM;
        const int mw = Sh::mma_index(warp);
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, DT_TOK);
            uint32_t gs = 0;         // stream index of the unit's first stage
            int qi = 0;
            uint32_t qph = 0;
            bool issued = false;  // any MMA of this thread
            for (;;) {
                if (!mbar_wait(&uq_full[qi], qph, abort_flag)) {
                    record_error(a.status, DEV_TIMEOUT_ACCUM_FREE);
                    *abort_flag = 1;
                    break;
                }
                const int u = uq[qi];
                if (u < 0) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)((qi * NM + mw) * DT_TOK);
                int nk;
                if (u < sc.up_units) {
                    const UpUnit x = up_unit(sc, u, a.F);
                    nk = x.kb1 - x.kb0;
                } else {
                    const DnUnit d = dn_unit(sc, u - sc.up_units, s_dnb);
                    nk = d.kb1 - d.kb0;
                }
                bool ok = true, first = true;
                // this thread's stages of the unit: stream indices g in [gs, gs + nst)
                // with g = mw mod NM; raw stage g mod RS (low-bit: A tile g mod AS)
                const uint32_t nst = (uint32_t)((nk + Sh::KPS - 1) / Sh::KPS);
                for (uint32_t g = gs + (uint32_t)((mw + NM - (int)(gs % NM)) % NM); g < gs + nst; g += NM) {
                    const int stage = (int)(g % RS), ast = (int)(g % DT_FP4_AS);
                    // low-bit: the A tile is in tensor memory once the block it came
                    // from has landed, so the token tile has too
                    if (FP4 ? !mbar_wait(&deq[ast], (g / DT_FP4_AS) & 1u, abort_flag)
                            : !mbar_wait(&full[stage], (g / RS) & 1u, abort_flag)) {
                        record_error(a.status, DEV_TIMEOUT_FULL_BARRIER);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = smem_u32(smem + Sh::B_OFF + stage * Sh::B_STRIDE);
                    if (FP4) {
                        const int nkb = min(Sh::KPS, nk - (int)(g - gs) * Sh::KPS);
                        const uint32_t at = tmem_base + (uint32_t)(DT_FP4_A_COL + ast * 32 * Sh::KPS);
                        for (int sub = 0; sub < nkb; ++sub)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_ta(d_tmem, at + sub * 32 + k * 8, smem_desc_sw128(sb + sub * DT_B_BYTES + k * 32),
                                       idesc, !first || sub != 0 || k != 0);
                    } else {
                        const uint32_t sa = smem_u32(smem + stage * Sh::A_STRIDE);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(d_tmem, smem_desc_sw128(sa + k * 32), smem_desc_sw128(sb + k * 32), idesc,
                                     !first || k != 0);
                    }
                    mma_commit(&empty[stage]);  // the raw stage (and low-bit: the A tile) is free
                    first = false;
                    issued = true;
                }
                gs += nst;
                if (!ok) break;
                mma_commit(&acc_full[qi]);  // MXFP4: also when this thread had no stage of the unit
                if (++qi == ACC) qi = 0, qph ^= 1;
            }
            if (issued) {
                // no MMA of this thread may still write tensor memory at teardown
                volatile int never = 0;
                mma_commit(&drain[mw]);
                mbar_wait(&drain[mw], 0, &never);
            }
        }
    } else if (warp < 6) {
        // ------------------------------ epilogue (warps 2..5) ------------------------------
        const int q = warp & 3;
        const int r = q * 32 + lane;                // accumulator row = weight row of the tile
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const int et = threadIdx.x - 64;            // 0..127 within the epilogue group
        if (et == 96) {
            // the down split ranges; only needed once the gate/up units are all
            // claimed, so they are computed here rather than in the prologue.  A
            // down unit reaches the MMA and epilogue roles only through the
            // producer, which waits for this barrier first.
            s_sdn = down_bounds(sc.total_kb, sc.ot, G, min(DT_MAX_DOWN_SPLITS, a.max_units / sc.ot), s_dnb);
            mbar_arrive(&s_bnd_bar);
        }
        int qi = 0;
        uint32_t qph = 0;
        uint32_t e_gs = 0;  // MXFP4: index in the stream of the unit's first stage
        for (;;) {
            // one thread waits (bounded) and tells the others, so that all 128
            // leave together and no named barrier below can hang
            if (et == 0) {
                int go = 1;
                if (!mbar_wait(&uq_full[qi], qph, abort_flag)) go = 0;
                else if (uq[qi] < 0) go = 2;
                else if (!mbar_wait(&acc_full[qi], qph, abort_flag)) go = 0;
                if (go == 0) {
                    record_error(a.status, DEV_TIMEOUT_ACCUM_BARRIER);
                    *abort_flag = 1;
                }
                bcast[1] = go;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int go = bcast[1];
            const int u = uq[qi];
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (go != 1) break;
            const bool is_up = u < sc.up_units;
            UpUnit ux;
            DnUnit dx;
            int tile, S, tbase, pslot, nk;
            if (is_up) { ux = up_unit(sc, u, a.F); tile = ux.tile; S = ux.S; tbase = 0; pslot = ux.pslot; nk = ux.kb1 - ux.kb0; }
            else {
                dx = dn_unit(sc, u - sc.up_units, s_dnb);
                tile = dx.tile; S = s_sdn; tbase = DT_TICKET_DOWN; pslot = a.max_units + tile * S; nk = dx.kb1 - dx.kb0;
            }
            tc_fence_after();
            uint32_t raw[16];
            float v[DT_TOK];
            {
                // the MMA threads' accumulators: the one holding the unit's stages
                // j, j + NM, j + 2 NM, ... is that of thread (e_gs + j) mod NM (its
                // stream indices are e_gs .. e_gs + nst - 1); they are added in the
                // order of j, which does not depend on where the unit fell in this
                // CTA's stream, so that the sum is the same bits on every run
#pragma unroll
                for (int t = 0; t < DT_TOK; ++t) v[t] = 0.0f;
                const int nst = (nk + Sh::KPS - 1) / Sh::KPS;  // stages of the unit
#pragma unroll
                for (int j = 0; j < Sh::NM; ++j) {
                    if (j >= nst) break;  // a unit of fewer stages than MMA threads
                    const int m = (int)((e_gs + (uint32_t)j) % Sh::NM);
                    tmem_ld16(tmem_base + lane_addr + (uint32_t)((qi * Sh::NM + m) * DT_TOK), raw);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < DT_TOK; ++t) v[t] += __uint_as_float(raw[t]);
                }
                e_gs += (uint32_t)nst;
            }

            bool finalize = true;
            if (S > 1) {
                // the partial of this split to global, one row of 128 floats per
                // token; the last split of the tile to arrive sums all of them in
                // split order
                const int split = is_up ? ux.s : dx.s;
                float *pt = a.partials + (size_t)T * 128 * pslot;
#pragma unroll
                for (int t = 0; t < DT_TOK; ++t)
                    if (t < T) pt[((size_t)split * T + t) * 128 + r] = v[t];
                // the named barrier orders the group's stores before one thread's
                // acquire-release ticket
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (et == 0) {
                    const int last = atom_acq_rel_add(&tickets[tbase + tile], 1) == S - 1;
                    if (last) tickets[tbase + tile] = 0;
                    bcast[2] = last;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                finalize = bcast[2] != 0;
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (finalize) {
#pragma unroll
                    for (int t = 0; t < DT_TOK; ++t) v[t] = 0.0f;
                    if (T <= 4) sum_partials<4, 8>(pt, S, T, r, v);
                    else sum_partials<16, 2>(pt, S, T, r, v);
                }
            }
            if (finalize) {
                // the tile to shared memory, so that the per-token loops below
                // need not be unrolled (row pitch 17: conflict-free by row)
#pragma unroll
                for (int t = 0; t < DT_TOK; ++t) xch[r * DT_EP_LD + t] = v[t];
                // 16 threads look up each token's routing weight for this group
                if (is_up && et < DT_TOK)
                    s_wt[et] = et < T ? group_weight(ux.g, et, sc.n_act, K, s_act, s_idx, s_w, s_gsh) : 0.0f;
                asm volatile("bar.sync 1, 128;" ::: "memory");
            }
            if (finalize && is_up) {
                // rows 0..63 are gate projections, rows 64..127 the matching up
                // projections.  All 128 threads: feature r % 64 for every other
                // token from r / 64.  Only the T real token rows of h' are written:
                // a row t >= T feeds only column t of the down accumulator, which
                // nothing reads.
                {
                    const int fr = r & 63;
                    const int f = ux.ft * 64 + fr;
                    const int e = ux.shared ? -1 : s_act[ux.g];
                    const float bg = (!ux.shared && a.gate_b) ? a.gate_b[(size_t)e * a.F + f] : 0.0f;
                    const float bu = (!ux.shared && a.up_b) ? a.up_b[(size_t)e * a.F + f] : 0.0f;
                    const bool swiglu = ux.shared || a.act == MOE_ACT_SWIGLU;
                    const size_t hbase = (size_t)ux.g * DT_TOK * a.Fmax + f;
#pragma unroll 1
                    for (int t = r >> 6; t < T; t += 2) {
                        const float gv = xch[fr * DT_EP_LD + t] + bg, uv = xch[(fr + 64) * DT_EP_LD + t] + bu;
                        float hval = swiglu ? activation<MOE_ACT_SWIGLU>(gv, uv, a.alpha, a.limit)
                                            : activation<MOE_ACT_CLAMP_GLU>(gv, uv, a.alpha, a.limit);
                        hval *= s_wt[t];
                        reinterpret_cast<__nv_bfloat16 *>(a.hp)[hbase + (size_t)t * a.Fmax] = __float2bfloat16_rn(hval);
                    }
                }
                // publish: h' of this tile is written (generic proxy) and will be
                // read by TMA (async proxy) in other CTAs
                fence_proxy_async_global();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (et == 0) red_release_add(&group_done[ux.g * DT_DONE_STRIDE], 1);
            } else if (finalize) {
                const int row = dx.tile * 128 + r;
                if (row < a.H) {
#pragma unroll 1
                    for (int t = 0; t < T; ++t) {
                        float o = xch[r * DT_EP_LD + t];
                        if (a.down_b)
                            for (int j = 0; j < K; ++j)
                                o += s_w[t * K + j] * a.down_b[(size_t)s_idx[t * K + j] * a.H + row];
                        const size_t oi = (size_t)t * a.H + row;
                        if (a.out_bf16) reinterpret_cast<__nv_bfloat16 *>(a.out)[oi] = __float2bfloat16_rn(o);
                        else reinterpret_cast<float *>(a.out)[oi] = o;
                    }
                }
            }
            // the accumulator and the queue slot are free again
            tc_fence_before();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (et == 0) mbar_arrive(&uq_empty[qi]);
            if (++qi == ACC) qi = 0, qph ^= 1;
        }
    } else if (FP4 && warp < 6 + DT_FP4_DQW) {
        // ------------------------------ low-bit dequantisation (warps 6 .. 5 + DQW) ------------------------------
        // Follows the units in queue order like the MMA threads.  DQG groups of
        // four warps take the stages in turn (by their index in the stream); in a
        // group, warp w widens the rows of its 32-lane quadrant w % 4, lane =
        // row, straight into the A tile in tensor memory (a warp reaches only
        // its own quadrant's lanes).  A tile is rewritten once the MMA
        // DT_FP4_AS stages back, its last reader, has completed (that stage's
        // release of its raw stage).  After a failed wait the loop keeps going
        // without work (every later wait fails fast on the abort flag) until the
        // producer's end marker, so the named barrier below always sees all the
        // warps.
        __shared__ int s_dq[2];
        const int dr = threadIdx.x - DT_THREADS;  // 0 .. 32 * DT_FP4_DQW - 1
        const int q = warp & 3, grp = (warp - 6) >> 2;
        const int row = q * 32 + lane;
        const uint32_t t_a = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)DT_FP4_A_COL;
        int qi = 0;
        uint32_t qph = 0;
        uint32_t gs = 0;  // stream index of the unit's first stage
        for (;;) {
            if (dr == 0) {
                int go = 1;
                if (!mbar_wait(&uq_full[qi], qph, abort_flag)) go = 0;
                else if (uq[qi] < 0) go = 2;
                if (go == 0) {
                    record_error(a.status, DEV_TIMEOUT_ACCUM_BARRIER);
                    *abort_flag = 1;
                }
                s_dq[0] = go;
                s_dq[1] = go == 1 ? uq[qi] : -1;
            }
            asm volatile("bar.sync 2, %0;" ::"n"(32 * DT_FP4_DQW) : "memory");
            const int go = s_dq[0], u = s_dq[1];
            asm volatile("bar.sync 2, %0;" ::"n"(32 * DT_FP4_DQW) : "memory");
            if (go != 1) break;
            int nk;
            if (u < sc.up_units) {
                const UpUnit x = up_unit(sc, u, a.F);
                nk = x.kb1 - x.kb0;
            } else {
                const DnUnit d = dn_unit(sc, u - sc.up_units, s_dnb);
                nk = d.kb1 - d.kb0;
            }
            // this group's stages of the unit: stream indices g in [gs, gs + nst) with
            // g = grp mod DQG; raw stage g mod RS, A tile g mod AS
            const uint32_t nst = (uint32_t)((nk + DT_FP4_KPS - 1) / DT_FP4_KPS);
            for (uint32_t g = gs + (uint32_t)((grp + DT_FP4_DQG - (int)(gs % DT_FP4_DQG)) % DT_FP4_DQG); g < gs + nst;
                 g += DT_FP4_DQG) {
                const int stage = (int)(g % RS), ast = (int)(g % DT_FP4_AS);
                bool ok = mbar_wait(&full[stage], (g / RS) & 1u, abort_flag);
                if (ok && g >= (uint32_t)DT_FP4_AS) {
                    // the tile's last reader, the MMA of stream stage g - AS, has completed
                    // (it released its raw stage)
                    const uint32_t gp = g - DT_FP4_AS;
                    ok = mbar_wait(&empty[gp % RS], (gp / RS) & 1u, abort_flag);
                }
                if (ok) {
                    tc_fence_after();
                    const int nkb = min(DT_FP4_KPS, nk - (int)(g - gs) * DT_FP4_KPS);
                    for (int sub = 0; sub < nkb; ++sub) {
                        const uint8_t *blk = smem + Sh::BLK_OFF + stage * Sh::BLK_STRIDE + sub * Sh::BLK;
                        const uint32_t col = (uint32_t)((ast * DT_FP4_KPS + sub) * 32);
                        uint32_t v[32];
                        lowbit_dequant_row<QF>(blk, row, fp4tab, v);
                        tmem_st32(t_a + col, v);
                    }
                    // the raw stage is refilled by a bulk copy (async proxy) once the
                    // MMA releases it: order these generic reads before that copy
                    fence_proxy_async_shared();
                    tmem_st_wait();
                } else if (!*abort_flag) {
                    record_error(a.status, DEV_TIMEOUT_FULL_BARRIER);
                    *abort_flag = 1;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&deq[ast]);
            }
            gs += nst;
            if (++qi == ACC) qi = 0, qph ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(Sh::TMEM_COLS));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static bool dec_encode(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                       bool f16 = false)
{
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
               dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool dectc_supported(const Layer &L, int T)
{
    return L.dectc != nullptr && T >= 1 && T <= DT_TOK;
}

static int dectc_groups_max(const Layer &L)
{
    const int routed = L.E < DT_TOK * L.K ? L.E : DT_TOK * L.K;
    return routed + (L.Fs > 0 ? 1 : 0);
}

size_t dectc_workspace(const Layer &L, size_t &hp_bytes, size_t &part_bytes, size_t &tab_bytes, size_t &ticket_bytes)
{
    hp_bytes = (size_t)dectc_groups_max(L) * DT_TOK * L.Fmax * 2;
    part_bytes = (size_t)L.num_sms * DT_UNITS_PER_CTA * 128 * DT_TOK * 4 * 2;  // gate/up and down partials
    tab_bytes = 16;
    ticket_bytes = (size_t)DT_COUNTERS * 4;
    return hp_bytes + part_bytes + tab_bytes + ticket_bytes;
}

int dectc_prepare(Layer &L)
{
    if ((long long)dectc_groups_max(L) * DT_DONE_STRIDE > DT_NEXT_UNIT - DT_GROUP_DONE) return -1;
    DecMaps *m = new (std::nothrow) DecMaps();
    if (!m) return -1;
    bool ok = dec_encode(&m->hp, L.dec_hp, L.Fmax, (uint64_t)dectc_groups_max(L) * DT_TOK, DT_TOK);
    if (L.qfmt != QF_NONE) {
        // the experts stream as packed low-bit blocks (bulk copies), not through tensor maps
        m->gate = m->up = m->down = m->hp;
    } else {
        // (the weight arrays hold wslots experts: every one, or the resident slots)
        ok = ok && dec_encode(&m->gate, L.gate_w, L.H, (uint64_t)L.wslots * L.F, 64) &&
             dec_encode(&m->up, L.up_w, L.H, (uint64_t)L.wslots * L.F, 64) &&
             dec_encode(&m->down, L.down_w, L.F, (uint64_t)L.wslots * L.H, 128);
    }
    if (ok && L.Fs) {
        ok = dec_encode(&m->sh_gate, L.sh_gate_w, L.H, L.Fs, 64) && dec_encode(&m->sh_up, L.sh_up_w, L.H, L.Fs, 64) &&
             dec_encode(&m->sh_down, L.sh_down_w, L.Fs, L.H, 128);
    } else if (ok) {
        m->sh_gate = m->gate;
        m->sh_up = m->up;
        m->sh_down = m->down;
    }
    if (ok)
        ok = cudaFuncSetAttribute(dec_experts_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)DtShape<0>::SMEM) == cudaSuccess &&
             cudaFuncSetAttribute(dec_experts_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)DtShape<1>::SMEM) == cudaSuccess &&
             cudaFuncSetAttribute(dec_experts_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)DtShape<2>::SMEM) == cudaSuccess;
    if (!ok) { delete m; return -1; }
    L.dectc = m;
    return 0;
}

void dectc_release(Layer &L)
{
    delete L.dectc;
    L.dectc = nullptr;
}

// which: 0 = router logits, 1 = selection + experts (writes out)
int launch_dectc(const Layer &L, const void *x, int T, void *out, int which, cudaStream_t s, int t0)
{
    if (which == 0) {
        DecRouteArgs r;
        r.x = (const __nv_bfloat16 *)x;
        r.router_w = (const __nv_bfloat16 *)L.router_w;
        r.router_b = L.router_b;
        r.logits = L.logits + (size_t)t0 * L.R;
        r.counters = L.dec_tickets;
        r.T = T; r.E = L.E; r.H = L.H; r.R = L.R;
        r.n_reset = dectc_groups_max(L);
        dec_route_kernel<<<L.R, 256, 0, s>>>(r);
        return 1;
    }
    DecMaps m = *L.dectc;
    if (!dec_encode(&m.x, x, L.H, (uint64_t)T, DT_TOK)) return -1;
    DecArgs a;
    a.logits = L.logits + (size_t)t0 * L.R;
    a.topk_idx = L.topk_idx + (size_t)t0 * L.K;
    a.topk_w = L.topk_w + (size_t)t0 * L.K;
    a.sh_gate = L.sh_gate + t0;
    a.counts = L.counts; a.active = L.active;
    a.slot_of = L.S > 0 ? L.slot_of : nullptr;
    a.accumulate = t0 > 0;
    a.meta = L.meta;
    a.gate_b = L.gate_b; a.up_b = L.up_b; a.down_b = L.down_b;
    a.hp = L.dec_hp;
    a.gu_fp4 = L.fp4_gu;
    a.dn_fp4 = L.fp4_dn;
    a.ot = (L.H + 127) / 128;
    a.partials = L.dec_partials;
    a.counters = L.dec_tickets;
    a.out = out;
    a.status = L.status;
    a.T = T; a.K = L.K; a.E = L.E; a.H = L.H; a.F = L.F; a.Fs = L.Fs; a.Fmax = L.Fmax; a.R = L.R;
    a.mode = L.cfg.router_mode; a.norm = L.cfg.norm_topk_prob; a.scale = L.cfg.weights_scale;
    a.act = L.cfg.act;
    a.out_bf16 = L.cfg.out_dtype == MOE_DT_BF16;
    a.alpha = L.cfg.act_alpha; a.limit = L.cfg.act_limit;
    a.max_units = L.num_sms * DT_UNITS_PER_CTA;
    a.wait_ns = L.wait_ns;
    a.inject = L.inject;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(L.qfmt == QF_Q4 ? DtShape<2>::THREADS : L.qfmt == QF_MXFP4 ? DtShape<1>::THREADS
                                                                                    : DtShape<0>::THREADS);
    cfg.dynamicSmemBytes = L.qfmt == QF_Q4 ? DtShape<2>::SMEM : L.qfmt == QF_MXFP4 ? DtShape<1>::SMEM
                                                                                 : DtShape<0>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = L.qfmt == QF_Q4      ? cudaLaunchKernelEx(&cfg, dec_experts_kernel<2>, m, a)
                          : L.qfmt == QF_MXFP4 ? cudaLaunchKernelEx(&cfg, dec_experts_kernel<1>, m, a)
                                               : cudaLaunchKernelEx(&cfg, dec_experts_kernel<0>, m, a);
    return e == cudaSuccess ? 1 : -1;
}

// ---------------------------------------------------------------------------
// MXFP4 packing for the decode kernel: each (row block, 64-wide K block) of a
// matrix becomes one contiguous block of LOWBIT_BLK_MXFP4 bytes, the codes as
// [2 halves][128 rows][16 B] (half h = the row's 32-element source block
// 2 kb + h) and then the scales as [2 halves][128 rows], so that a warp
// reading one half of 32 consecutive rows reads 512 contiguous bytes.
// gate/up: 64 gate rows then the 64 matching up rows of the de-interleaved
// gate_up; down: 128 output rows, rows past H zero (code 0 is the value 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fp4_pack_row(uint8_t *blk, int trow, const uint8_t *src_blocks,
                                             const uint8_t *src_scales)
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        reinterpret_cast<uint4 *>(blk + (h * 128 + trow) * 16)[0] =
            src_blocks ? reinterpret_cast<const uint4 *>(src_blocks)[h] : make_uint4(0, 0, 0, 0);
        blk[128 * 32 + h * 128 + trow] = src_scales ? src_scales[h] : 127;
    }
}

__global__ void pack_fp4_gate_up_kernel(const uint8_t *blocks, const uint8_t *scales, int E, int F, int H,
                                        uint8_t *out)
{
    const int nkb = H / 64, nb = H / 32;
    const size_t n = (size_t)E * 2 * F * nkb;  // one (source row, K block) each
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / nkb;               // interleaved row of [E][2F]
        const int kb = (int)(i - row * nkb);
        const int e = (int)(row / (2 * F)), rr = (int)(row - (size_t)e * 2 * F);
        const int f = rr >> 1, up = rr & 1;
        const size_t blk = ((size_t)e * (F / 64) + f / 64) * nkb + kb;
        fp4_pack_row(out + blk * LOWBIT_BLK_MXFP4, up * 64 + (f & 63), blocks + (row * nb + 2 * kb) * 16,
                     scales + row * nb + 2 * kb);
    }
}

__global__ void pack_fp4_down_kernel(const uint8_t *blocks, const uint8_t *scales, int E, int F, int H, uint8_t *out)
{
    const int nkb = F / 64, nb = F / 32, ot = (H + 127) / 128;
    const size_t n = (size_t)E * ot * 128 * nkb;  // one (padded output row, K block) each
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t prow = i / nkb;               // [E][ot*128]
        const int kb = (int)(i - prow * nkb);
        const int e = (int)(prow / ((size_t)ot * 128)), h = (int)(prow - (size_t)e * ot * 128);
        const size_t blk = ((size_t)e * ot + h / 128) * nkb + kb;
        const size_t row = (size_t)e * H + h;
        fp4_pack_row(out + blk * LOWBIT_BLK_MXFP4, h & 127, h < H ? blocks + (row * nb + 2 * kb) * 16 : nullptr,
                     h < H ? scales + row * nb + 2 * kb : nullptr);
    }
}

// Q4: the same block layout with a binary16 scale per row and half.  The
// codes of each record are rearranged so that the eight elements 8q .. 8q+7
// of a half form 32-bit word q, element 8q + i in nibble q4_nibble_of(i)
// (evens in nibbles 0..3, odds in 4..7; see q4_to_bf16x8).  A record's byte
// j holds elements j (low nibble) and j + 16.  Rows past H get scale 0
// (value 0).
__device__ __forceinline__ void q4_pack_row(uint8_t *blk, int trow, const uint8_t *rec0, const uint8_t *rec1)
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint8_t *rec = h ? rec1 : rec0;
        uint32_t words[4] = {0u, 0u, 0u, 0u};
        uint16_t d = 0;
        if (rec) {
            d = (uint16_t)(rec[0] | (rec[1] << 8));
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const uint32_t c = e < 16 ? (rec[2 + e] & 15u) : (rec[2 + e - 16] >> 4);
                words[e >> 3] |= c << (4 * q4_nibble_of(e & 7));
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) words[q] = 0x88888888u;
        }
        reinterpret_cast<uint4 *>(blk + (h * 128 + trow) * 16)[0] = make_uint4(words[0], words[1], words[2], words[3]);
        reinterpret_cast<uint16_t *>(blk + LOWBIT_CODE_BYTES)[h * 128 + trow] = d;
    }
}

// gate/up rows come from an interleaved [E][2F] tensor (gate = even rows) or
// from separate gate and up tensors [E][F]; records of H/32 blocks of 18 bytes
__global__ void pack_q4_gate_up_kernel(const uint8_t *gate_up, const uint8_t *gate, const uint8_t *up, int E, int F,
                                       int H, uint8_t *out)
{
    const int nkb = H / 64, nb = H / 32;
    const size_t n = (size_t)E * 2 * F * nkb;  // one (gate/up row, K block) each
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / nkb;               // [E][2F]: (feature, gate / up) pairs
        const int kb = (int)(i - row * nkb);
        const int e = (int)(row / (2 * F)), rr = (int)(row - (size_t)e * 2 * F);
        const int f = rr >> 1, isup = rr & 1;
        const uint8_t *src = gate_up ? gate_up + ((size_t)e * 2 * F + 2 * f + isup) * nb * 18
                                     : (isup ? up : gate) + ((size_t)e * F + f) * nb * 18;
        const size_t blk = ((size_t)e * (F / 64) + f / 64) * nkb + kb;
        q4_pack_row(out + blk * LOWBIT_BLK_Q4, isup * 64 + (f & 63), src + 2 * kb * 18, src + (2 * kb + 1) * 18);
    }
}

__global__ void pack_q4_down_kernel(const uint8_t *down, int E, int F, int H, uint8_t *out)
{
    const int nkb = F / 64, nb = F / 32, ot = (H + 127) / 128;
    const size_t n = (size_t)E * ot * 128 * nkb;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t prow = i / nkb;
        const int kb = (int)(i - prow * nkb);
        const int e = (int)(prow / ((size_t)ot * 128)), h = (int)(prow - (size_t)e * ot * 128);
        const size_t blk = ((size_t)e * ot + h / 128) * nkb + kb;
        const uint8_t *src = h < H ? down + ((size_t)e * H + h) * nb * 18 : nullptr;
        q4_pack_row(out + blk * LOWBIT_BLK_Q4, h & 127, src ? src + 2 * kb * 18 : nullptr,
                    src ? src + (2 * kb + 1) * 18 : nullptr);
    }
}

size_t dectc_fp4_bytes(const Layer &L, bool gate_up)
{
    const size_t ot = (L.H + 127) / 128;
    const size_t blk = L.qfmt == QF_Q4 ? LOWBIT_BLK_Q4 : LOWBIT_BLK_MXFP4;
    return gate_up ? (size_t)L.E * (L.F / 64) * (L.H / 64) * blk : (size_t)L.E * ot * (L.F / 64) * blk;
}

int dectc_pack_q4(Layer &L, const uint8_t *gate_up, const uint8_t *gate, const uint8_t *up, const uint8_t *down)
{
    pack_q4_gate_up_kernel<<<4 * L.num_sms, 256>>>(gate_up, gate, up, L.E, L.F, L.H, L.fp4_gu);
    pack_q4_down_kernel<<<4 * L.num_sms, 256>>>(down, L.E, L.F, L.H, L.fp4_dn);
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}

int dectc_pack_fp4(Layer &L, const uint8_t *gu_blocks, const uint8_t *gu_scales, const uint8_t *dn_blocks,
                   const uint8_t *dn_scales)
{
    pack_fp4_gate_up_kernel<<<4 * L.num_sms, 256>>>(gu_blocks, gu_scales, L.E, L.F, L.H, L.fp4_gu);
    pack_fp4_down_kernel<<<4 * L.num_sms, 256>>>(dn_blocks, dn_scales, L.E, L.F, L.H, L.fp4_dn);
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}

}  // namespace moe
