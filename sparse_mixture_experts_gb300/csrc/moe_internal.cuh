// moe_internal.cuh -- layer object, device helpers and kernel entry points
// shared by the translation units of libmoe.  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// device status word: kernels record the first error they hit here
// ---------------------------------------------------------------------------
enum DeviceError : int {
    DEV_OK = 0,
    DEV_TIMEOUT_FULL_BARRIER = 1,   // producer->MMA smem stage never filled
    DEV_TIMEOUT_EMPTY_BARRIER = 2,  // MMA->producer smem stage never drained
    DEV_TIMEOUT_ACCUM_BARRIER = 3,  // MMA->epilogue accumulator never ready
    DEV_TIMEOUT_ACCUM_FREE = 4,     // epilogue->MMA accumulator never released
    DEV_BAD_TILE = 5,               // a tile descriptor outside the problem
    DEV_TIMEOUT_GRID_BARRIER = 6,   // a block of the cooperative decode kernel never arrived
    DEV_TIMEOUT_DEPENDENCY = 7,     // a group's activations never completed (weight-streaming decode kernel)
    DEV_TIMEOUT_INJECTED = 8,       // the test-only injected wait ran out (tensor-core GEMMs)
    DEV_NOT_RESIDENT = 9,           // a selected expert had no slot (expert residency)
};

// Groups of rows a grouped kernel walks over: the routed experts that
// received at least one token (ascending expert index), then the shared
// expert (all tokens) when the layer has one.
constexpr int SEL_TOK = 16;  // tokens per selection block (a grouping chunk)

struct RouteMeta {
    int ticket;       // arrival counter of the grouping kernel (reset by its last block)
    int n_active;     // routed experts with count > 0
    int n_up_tiles;   // tensor-core tiles of the gate/up GEMM
    int n_down_tiles; // tensor-core tiles of the down GEMM
    int n_pairs;      // T * k
    int pad[3];
};

struct TensorMaps;  // defined in expert_tc.cu

// the routed experts' storage
enum QuantFormat : int {
    QF_NONE = 0,   // w_dtype (bf16 or fp32) tensors
    QF_MXFP4 = 1,  // MXFP4 blocks, packed (lowbit.cuh)
    QF_Q4 = 2,     // Q4 records, packed (lowbit.cuh)
};

struct Layer {
    moe_config cfg{};
    int device = 0;
    int num_sms = 0;
    int path = MOE_PATH_AUTO;
    bool tc_capable = false;
    int E = 0, H = 0, F = 0, Fs = 0, K = 0, R = 0;  // R = router rows (E, +1 for the shared gate)
    int Fmax = 0;
    int Tmax = 0;
    size_t wbytes = 0;  // element size of weights / activations

    // weights, library-owned, [out][in]
    void *router_w = nullptr;  // [R][H]; row E = shared gate vector when Fs > 0
    float *router_b = nullptr; // [E]
    void *gate_w = nullptr;    // [E][F][H]
    void *up_w = nullptr;      // [E][F][H]
    float *gate_b = nullptr;   // [E][F]
    float *up_b = nullptr;     // [E][F]
    void *down_w = nullptr;    // [E][H][F]
    float *down_b = nullptr;   // [E][H]
    void *sh_gate_w = nullptr; // [Fs][H]
    void *sh_up_w = nullptr;   // [Fs][H]
    void *sh_down_w = nullptr; // [H][Fs]

    // workspace, sized for Tmax tokens
    float *logits = nullptr;   // [Tmax][R]
    float *router_parts = nullptr;  // [TC_ROUTER_MAX_SPLITS][Tmax][R] partial logits of the split router GEMM
    int *topk_idx = nullptr;   // [Tmax][K]
    float *topk_w = nullptr;   // [Tmax][K]
    float *sh_gate = nullptr;  // [Tmax]
    int *counts = nullptr;     // [E]
    int *offsets = nullptr;    // [E + 1]
    int *expert_rows = nullptr;// [Tmax*K] pair ids t*K+slot sorted by expert (from offsets[e]), ascending t
    int *chunk_hist = nullptr; // [E][hist_pitch] picks per chunk of SEL_TOK tokens, then where they start
    int *pair_rank = nullptr;  // [Tmax][K] rank of each pick among its chunk's picks of the same expert
    int hist_pitch = 0;        // chunks per expert row (>= ceil(Tmax / SEL_TOK), a multiple of 4)
    int *active = nullptr;     // [E]
    RouteMeta *meta = nullptr;
    void *h = nullptr;         // [Tmax*K + Tmax][Fmax] activations (routed rows sorted by expert, then shared)
    void *xp = nullptr;        // [Tmax*K + Tmax][H] x rows gathered in expert order, then x (tensor-core path)
    float *ys = nullptr;       // [Tmax][K+1][H] weighted expert outputs per (token, slot), fp32
    int qfmt = 0;              // QF_NONE, or the routed experts' low-bit format (fp4_gu / fp4_dn; gate_w,
                               // up_w, down_w unused)
    int *gfirst = nullptr;     // [5][E + 2] per group: first gate/up tile (and the total), first down tile
                               // (and the total), expert (E = shared), rows, first row in the sorted buffers
    int *status = nullptr;     // DeviceError
    int *never = nullptr;      // a device word that stays 0 (what fault injection waits for)
    unsigned long long wait_ns = 1000000000ull;  // bound of a wait on another block (moe_set_wait_limit)
    int inject = 0;            // test-only: the next forwards wait for what never happens
    unsigned *gbar = nullptr;  // [2] grid-barrier arrivals / generation (decode kernel)
    int decode_grid = 0;       // blocks of the cooperative decode kernel (0 = unavailable)
    void *x_stage = nullptr;   // [Tmax][H] for moe_forward_host
    void *out_stage = nullptr; // [Tmax][H]
    // moe_forward_host: the copy of x in runs on a stream of the layer's own,
    // ordered after the previous forward's reads of x_stage (x_free) and
    // before this forward (x_ready), so that it overlaps the work before it
    cudaStream_t h2d_stream = nullptr;
    cudaEvent_t x_ready = nullptr, x_free = nullptr;
    TensorMaps *tmaps = nullptr;  // host copy of the tensor maps (tensor-core path)
    // weight-streaming tensor-core decode path
    struct DecMaps *dectc = nullptr;
    void *dec_hp = nullptr;          // [groups_max*16][Fmax] bf16: routing-weighted activations
    float *dec_partials = nullptr;   // split-K partial sums
    float *dec_wtab = nullptr;       // [groups_max][16] routing weight of token t for group g
    int *dec_tickets = nullptr;      // per-tile arrival counters
    // MXFP4 experts: codes and scales packed per (row block, 64-wide K block)
    // so that a pipeline stage is one contiguous copy; both tensor-core paths
    // widen them to bf16 on chip
    uint8_t *fp4_gu = nullptr;       // [E][F/64][H/64] packed low-bit blocks (128 rows: 64 gate, 64 up)
    uint8_t *fp4_dn = nullptr;       // [E][ceil(H/128)][F/64] packed low-bit blocks
    // expert residency (cfg.resident_experts = S > 0): the routed experts'
    // weights in pinned host memory, and gate_w / up_w / down_w (or fp4_gu /
    // fp4_dn) holding S experts, one per slot
    int S = 0;                       // slots (0: every routed expert resident)
    int wslots = 0;                  // experts the device weight arrays hold (S, or E)
    int n_regions = 0;               // per-expert weight regions: 3 (gate, up, down) or 2 (low-bit)
    void *host_w[3] = {};            // pinned host copies, [E] experts each
    size_t region_bytes[3] = {};     // bytes per expert of each region
    void *dev_region[3] = {};        // the device slot arrays of the regions, [S] experts each
    int *slot_of = nullptr;          // [E] slot holding each expert, -1 if none
    int *expert_of = nullptr;        // [S] expert held by each slot, -1 if none
    unsigned *last_used = nullptr;   // [S] chunk stamp of each slot's last use
    int *res_jobs = nullptr;         // [1 + 2S] copies of the current chunk: count, (expert, slot) pairs
    unsigned long long *res_stats = nullptr;  // [4] hits, misses, bytes copied, chunks

    // per-kernel timing (moe_timing_enable / moe_timing_read)
    int timing_max = 0;         // forwards recorded per window; 0 = off
    int timing_recorded = 0;    // forwards recorded in the current window
    int timing_pairs = 0;       // event pairs used in the current window
    std::vector<cudaEvent_t> timing_events;  // 2 per pair
    std::vector<int> timing_kind;            // moe_kernel_kind per pair

    std::vector<void *> allocations;
    size_t device_bytes = 0;
    int last_T = 0;
    int last_launches = 0;
    int last_grouped = 0;       // 1: the last forward ran a grouped path (tensor-core or CUDA-core stream)
};

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// logistic function with the fast exponential and the fast (approximate)
// reciprocal: a few fp32 ulps, far below the bf16 rounding of the activations
// that follows on every bf16 path (an IEEE division here cost the gate/up
// epilogue about half of its time); 1 / inf gives 0 for very negative z
__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// routed-expert activation; ACT = moe_act
template <int ACT>
__device__ __forceinline__ float activation(float gate, float up, float alpha, float limit)
{
    if (ACT == MOE_ACT_SWIGLU) {
        return gate * sigmoidf_(gate) * up;
    } else {
        float g = fminf(gate, limit);
        float u = fminf(fmaxf(up, -limit), limit);
        return (u + 1.0f) * g * sigmoidf_(alpha * g);
    }
}

template <typename T> struct Vec;  // 16-byte vector of T
template <> struct Vec<float> {
    static constexpr int N = 4;
    float v[4];
    __device__ __forceinline__ void load(const float *p) {
        float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    }
    __device__ __forceinline__ void load_stream(const float *p) {
        float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    float v[8];
    __device__ __forceinline__ void unpack(uint4 a) {
        v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
        v[4] = bf16_lo(a.z); v[5] = bf16_hi(a.z); v[6] = bf16_lo(a.w); v[7] = bf16_hi(a.w);
    }
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
        unpack(__ldg(reinterpret_cast<const uint4 *>(p)));
    }
    __device__ __forceinline__ void load_stream(const __nv_bfloat16 *p) {
        unpack(__ldcs(reinterpret_cast<const uint4 *>(p)));
    }
};

__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Selection by one warp for NT tokens at once: lane j < k ends with the j-th
// pick of each token (descending logit, lower expert index on equal logits)
// and its routing weight.  Each lane holds NQ >= ceil(E/32) logits in
// registers (expert lane + 32 q).
//
// For NQ <= 8 every lane first sorts its candidates by a 64-bit key (the
// logit's order-preserving bit pattern above the complemented expert index),
// then each pick is two warp-wide integer max reductions over the lanes'
// heads (the larger logit, then among equal logits the lower index) and the
// winning lane pops its head.  For larger NQ each pick rescans the lane's
// candidates and reduces with shuffles.  Both orders are the same total order
// (value descending, index ascending), so the picks are identical.  -0 and
// +0 compare equal, as they do for the scan.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t logit_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;  // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int N>
__device__ __forceinline__ void sort_desc(unsigned long long (&c)[N])
{
    // bitonic network: every index is a compile-time constant, so c stays in registers
#pragma unroll
    for (int k = 2; k <= N; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int p = i ^ j;
                if (p > i) {
                    const unsigned long long x = c[i], y = c[p];
                    const bool sw = ((i & k) == 0) ? (x < y) : (x > y);
                    c[i] = sw ? y : x;
                    c[p] = sw ? x : y;
                }
            }
}

template <int NQ, int NT>
__device__ __forceinline__ void warp_topk(const float *const (&l)[NT], int E, int K, int mode, int norm, float scale,
                                          int lane, int (&sel_i)[NT], float (&sel_v)[NT], float (&w)[NT])
{
    float v[NT][NQ];
#pragma unroll
    for (int s = 0; s < NT; ++s)
#pragma unroll
        for (int q = 0; q < NQ; ++q) v[s][q] = (lane + 32 * q < E) ? __ldcg(l[s] + lane + 32 * q) : -INFINITY;

    // softmax over all E is only needed when the picks are not renormalised
    const bool need_z = mode == MOE_ROUTER_SOFTMAX_TOPK && !norm;
    float z[NT];
    if (need_z) {
#pragma unroll
        for (int s = 0; s < NT; ++s) {
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < NQ; ++q) mx = fmaxf(mx, v[s][q]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float zs = 0.0f;
#pragma unroll
            for (int q = 0; q < NQ; ++q) zs += (lane + 32 * q < E) ? __expf(v[s][q] - mx) : 0.0f;
            z[s] = warp_sum(zs);
        }
    }

    constexpr bool SORTED = NQ <= 8;
    unsigned long long c[NT][SORTED ? NQ : 1];
    uint32_t avail[NT];  // scan path: bit q set while candidate lane + 32 q is in range and not taken
#pragma unroll
    for (int s = 0; s < NT; ++s) {
        avail[s] = 0u;
#pragma unroll
        for (int q = 0; q < NQ; ++q) avail[s] |= (lane + 32 * q < E) ? (1u << q) : 0u;
    }
    if constexpr (SORTED) {
#pragma unroll
        for (int s = 0; s < NT; ++s) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const uint32_t idx = lane + 32 * q;
                c[s][q] = idx < (uint32_t)E ? ((unsigned long long)logit_key(v[s][q]) << 32) | (0xffffffffu - idx)
                                            : 0ull;
            }
            sort_desc<NQ>(c[s]);
        }
    }

    float top[NT], esum[NT], ex[NT];
#pragma unroll
    for (int s = 0; s < NT; ++s) {
        sel_i[s] = -1;
        sel_v[s] = 0.0f;
        esum[s] = 0.0f;
        ex[s] = 0.0f;
        top[s] = 0.0f;
    }
    for (int j = 0; j < K; ++j) {
        float bv[NT];
        int bi[NT];
        if constexpr (SORTED) {
            uint32_t hk[NT], hl[NT], m1[NT], m2[NT];
#pragma unroll
            for (int s = 0; s < NT; ++s) {
                hk[s] = (uint32_t)(c[s][0] >> 32);
                hl[s] = (uint32_t)c[s][0];
                m1[s] = __reduce_max_sync(0xffffffffu, hk[s]);
            }
#pragma unroll
            for (int s = 0; s < NT; ++s) m2[s] = __reduce_max_sync(0xffffffffu, hk[s] == m1[s] ? hl[s] : 0u);
#pragma unroll
            for (int s = 0; s < NT; ++s) {
                if (hk[s] == m1[s] && hl[s] == m2[s]) {  // this lane's head was picked
#pragma unroll
                    for (int q = 0; q + 1 < NQ; ++q) c[s][q] = c[s][q + 1];
                    c[s][NQ - 1] = 0ull;
                }
                bv[s] = key_logit(m1[s]);
                bi[s] = (int)(0xffffffffu - m2[s]);
            }
        } else {
#pragma unroll
            for (int s = 0; s < NT; ++s) {
                // lane-local best among the candidates not yet taken (ascending q:
                // a later q never beats an equal earlier one)
                int bq = -1;
                bv[s] = -INFINITY;
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    if (((avail[s] >> q) & 1u) && (bq < 0 || v[s][q] > bv[s])) { bv[s] = v[s][q]; bq = q; }
                bi[s] = bq < 0 ? 0x7fffffff : lane + 32 * bq;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int s = 0; s < NT; ++s) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv[s], o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi[s], o);
                    if (ov > bv[s] || (ov == bv[s] && oi < bi[s])) { bv[s] = ov; bi[s] = oi; }
                }
            }
#pragma unroll
            for (int s = 0; s < NT; ++s)
                if ((bi[s] & 31) == lane) avail[s] &= ~(1u << (bi[s] >> 5));  // taken
        }
        // every lane sees each pick, so each keeps the running sum of exp(pick - first pick)
#pragma unroll
        for (int s = 0; s < NT; ++s) {
            if (j == 0) top[s] = bv[s];
            const float e = __expf(bv[s] - top[s]);
            esum[s] += e;
            if (lane == j) { sel_i[s] = bi[s]; sel_v[s] = bv[s]; ex[s] = e; }
        }
    }
#pragma unroll
    for (int s = 0; s < NT; ++s) {
        if (lane >= K) w[s] = 0.0f;
        else if (mode == MOE_ROUTER_SOFTMAX_TOPK) w[s] = (need_z ? ex[s] / z[s] : ex[s] / esum[s]) * scale;
        else w[s] = ex[s] / esum[s];
    }
}

template <int NT>
__device__ __forceinline__ void warp_topk_any(const float *const (&l)[NT], int E, int K, int mode, int norm,
                                              float scale, int lane, int (&sel_i)[NT], float (&sel_v)[NT],
                                              float (&w)[NT])
{
    const int nq = (E + 31) / 32;
    if (nq <= 1) warp_topk<1, NT>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 2) warp_topk<2, NT>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 4) warp_topk<4, NT>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 8) warp_topk<8, NT>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 16) warp_topk<16, NT>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else warp_topk<32, NT>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
}

// one token per warp
__device__ __forceinline__ void warp_select_any(const float *l, int E, int K, int mode, int norm, float scale, int lane,
                                                int &sel_i, float &sel_v, float &w)
{
    const float *ls[1] = {l};
    int i[1];
    float v[1], ww[1];
    warp_topk_any<1>(ls, E, K, mode, norm, scale, lane, i, v, ww);
    sel_i = i[0];
    sel_v = v[0];
    w = ww[0];
}

// two tokens per warp (independent register sets, so their load latencies and
// dependent reductions overlap)
__device__ __forceinline__ void warp_select2_any(const float *la, const float *lb, int E, int K, int mode, int norm,
                                                 float scale, int lane, int (&sel_i)[2], float (&sel_v)[2],
                                                 float (&w)[2])
{
    const float *ls[2] = {la, lb};
    warp_topk_any<2>(ls, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
}

__device__ __forceinline__ void record_error(int *status, int code)
{
    atomicCAS(status, 0, code);
}

// message returned by moe_last_error() on this thread
void set_last_error(const char *msg);

// ---------------------------------------------------------------------------
// host-side launchers (each returns the number of kernels it launched, or -1)
// ---------------------------------------------------------------------------
int launch_router(const Layer &L, const void *x, int T, cudaStream_t s);
// with splits > 1, first adds the router's partial logits in split order
int launch_select(const Layer &L, int T, int splits, cudaStream_t s);
int launch_group(const Layer &L, int T, bool build_tiles, cudaStream_t s);
// positions of the picks in expert order; with rows, also gathers x into xp
int launch_scatter(const Layer &L, const void *x, int T, bool rows, cudaStream_t s);
// which: 0 = gate/up + activation, 1 = down + routing weight
int launch_experts_stream(const Layer &L, const void *x, int T, int which, cudaStream_t s);
int launch_combine(const Layer &L, int T, void *out, cudaStream_t s);

// fused decode kernel (decode.cu)
int decode_prepare(Layer &L);
bool decode_supported(const Layer &L, int T);
int launch_decode(const Layer &L, const void *x, int T, void *out, cudaStream_t s);

// weight-streaming tensor-core decode path (decode_tc.cu)
bool dectc_supported(const Layer &L, int T);
size_t dectc_workspace(const Layer &L, size_t &hp_bytes, size_t &part_bytes, size_t &tab_bytes, size_t &ticket_bytes);
int dectc_prepare(Layer &L);
// MXFP4 layers: pack the expert codes and scales for the decode kernel (from the
// caller's blocks and scales already on the device); 0 on success
size_t dectc_fp4_bytes(const Layer &L, bool gate_up);  // packed MXFP4 bytes of gate/up or down
int dectc_pack_fp4(Layer &L, const uint8_t *gu_blocks, const uint8_t *gu_scales, const uint8_t *dn_blocks,
                   const uint8_t *dn_scales);
// expert residency (residency.cu): move the routed experts' weights to pinned
// host memory and keep S slots on the device (at create, after the weights are
// final); per chunk of a forward, assign slots and copy the misses
moe_status residency_setup(Layer &L);
void residency_release(Layer &L);
int launch_residency(const Layer &L, const float *logits, int T, cudaStream_t s);
moe_status residency_read(Layer &L, int32_t *expert_of, int64_t *stats);
// Q4 layers: pack the records (gate/up interleaved, or gate and up apart) on the device; 0 on success
int dectc_pack_q4(Layer &L, const uint8_t *gate_up, const uint8_t *gate, const uint8_t *up, const uint8_t *down);
void dectc_release(Layer &L);
// which: 0 = router logits, 1 = selection + gate/up + down (writes out)
// t0: the chunk's first token within the forward (the logits and routing
// outputs of the chunk go to that offset; the expert counts accumulate)
int launch_dectc(const Layer &L, const void *x, int T, void *out, int which, cudaStream_t s, int t0 = 0);
constexpr int RESIDENT_CHUNK = 16;  // tokens per chunk of a layer with streamed experts

// tensor-core path (expert_tc.cu)
bool tc_supported(const Layer &L, std::string &why);
int tc_prepare(Layer &L);  // tensor maps over the layer's weights/workspace; 0 on success
void tc_release(Layer &L);
// which: 1 = gate/up GEMM + activation, 2 = down GEMM + weight (the token rows are gathered by launch_scatter)
int launch_experts_tc(const Layer &L, const void *x, int T, int which, cudaStream_t s);
int launch_tc_router(const Layer &L, const void *x, int T, cudaStream_t s);
int tc_router_splits(const Layer &L, int T);  // K ranges the tensor-core router uses for T tokens

constexpr int MAX_LAUNCHES_PER_FORWARD = 8;

// tile geometry of the tensor-core path (used by the grouping kernel)
constexpr int TC_BM = 128;       // token rows per tile
constexpr int TC_BN_UP = 256;    // gate/up tile: 128 gate + 128 up columns -> 128 h columns
constexpr int TC_BN_DOWN = 256;  // down tile: output columns
constexpr int TC_BK = 64;        // K elements per pipeline stage (128 bytes of bf16)
constexpr int TC_ROUTER_MAX_SPLITS = 4;  // K ranges of the tensor-core router GEMM
// low-bit experts: a tile is 256 token rows (two M = 128 halves sharing one
// widened weight tile, so that each weight block is widened once per 256
// rows) by one packed block of 128 weight rows (64 gate + 64 up features, or
// 128 down output columns)
constexpr int TC_LB_TM = 256;
constexpr int TC_LB_BN = 128;

// Low-bit layers take 256-row tiles (two M halves sharing each widened weight
// block) when a forward's routed experts have more than 128 rows on average
// (T k pairs over min(E, T k) experts), else 128-row tiles against two packed
// blocks, which halve the stages where the second half would stay empty.
inline bool tc_lowbit_two_halves(const Layer &L, int T)
{
    const long long pairs = (long long)T * L.K;
    const long long groups = pairs < L.E ? pairs : L.E;
    return L.qfmt != QF_NONE && pairs > 128LL * groups;
}

// token rows, gate/up features and down output columns per tile of the
// expert GEMMs of a forward of T tokens
struct TcGeometry {
    int tm, tnu, tnd;
};
inline TcGeometry tc_geometry(const Layer &L, int T)
{
    return tc_lowbit_two_halves(L, T) ? TcGeometry{TC_LB_TM, TC_LB_BN / 2, TC_LB_BN}
                                      : TcGeometry{TC_BM, TC_BN_UP / 2, TC_BN_DOWN};
}

}  // namespace moe
