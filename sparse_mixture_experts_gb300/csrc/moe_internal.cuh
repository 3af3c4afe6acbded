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
};

// Groups of rows a grouped kernel walks over: the routed experts that
// received at least one token (ascending expert index), then the shared
// expert (all tokens) when the layer has one.
struct RouteMeta {
    int ticket;       // arrival counter of the grouping kernel (reset by its last block)
    int n_active;     // routed experts with count > 0
    int n_up_tiles;   // tensor-core tiles of the gate/up GEMM
    int n_down_tiles; // tensor-core tiles of the down GEMM
    int n_pairs;      // T * k
    int pad[3];
};

// Tensor-core tile descriptor: group g (expert index, or E for the shared
// expert), first row m0 within the group, first output column n0.
struct TileDesc {
    int g;
    int m0;
    int n0;
    int pad;
};

struct TensorMaps;  // defined in expert_tc.cu

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
    int *topk_idx = nullptr;   // [Tmax][K]
    float *topk_w = nullptr;   // [Tmax][K]
    float *sh_gate = nullptr;  // [Tmax]
    int *counts = nullptr;     // [E]
    int *offsets = nullptr;    // [E + 1]
    int *expert_rows = nullptr;// [E][Tmax] pair ids t*K+slot, ascending t
    int *active = nullptr;     // [E]
    RouteMeta *meta = nullptr;
    void *h = nullptr;         // [Tmax*K + Tmax][Fmax] activations (routed rows sorted by expert, then shared)
    void *xp = nullptr;        // [Tmax*K + Tmax][H] x rows gathered in expert order, then x (tensor-core path)
    void *ys = nullptr;        // [Tmax][K+1][H] weighted expert outputs per (token, slot), weight dtype
    TileDesc *up_tiles = nullptr;
    TileDesc *down_tiles = nullptr;
    int max_up_tiles = 0, max_down_tiles = 0;
    int *status = nullptr;     // DeviceError
    unsigned *gbar = nullptr;  // [2] grid-barrier arrivals / generation (decode kernel)
    int decode_grid = 0;       // blocks of the cooperative decode kernel (0 = unavailable)
    void *x_stage = nullptr;   // [Tmax][H] for moe_forward_host
    void *out_stage = nullptr; // [Tmax][H]
    TensorMaps *tmaps = nullptr;  // host copy of the tensor maps (tensor-core path)
    // weight-streaming tensor-core decode path
    struct DecMaps *dectc = nullptr;
    void *dec_hp = nullptr;          // [groups_max*16][Fmax] bf16: routing-weighted activations
    float *dec_partials = nullptr;   // split-K partial sums
    float *dec_wtab = nullptr;       // [groups_max][16] routing weight of token t for group g
    int *dec_tickets = nullptr;      // per-tile arrival counters

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
};

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + __expf(-z)); }

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
// selection for one token by one warp: lane j < k ends with the j-th pick
// (descending logit, lower index on ties) and its routing weight.  Each lane
// holds NQ >= ceil(E/32) logits in registers (expert lane + 32 q).
// ---------------------------------------------------------------------------
template <int NQ>
__device__ __forceinline__ void warp_select(const float *l, int E, int K, int mode, int norm, float scale, int lane,
                                            int &sel_i, float &sel_v, float &w)
{
    float v[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) v[q] = (lane + 32 * q < E) ? __ldcg(l + lane + 32 * q) : -INFINITY;
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < NQ; ++q) mx = fmaxf(mx, v[q]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float z = 0.0f;
    if (mode == MOE_ROUTER_SOFTMAX_TOPK) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) z += (lane + 32 * q < E) ? __expf(v[q] - mx) : 0.0f;
        z = warp_sum(z);
    }
    sel_i = -1;
    sel_v = 0.0f;
    for (int j = 0; j < K; ++j) {
        // lane-local best (ascending q: a later q never beats an equal earlier one)
        float bv = v[0];
        int bq = 0;
#pragma unroll
        for (int q = 1; q < NQ; ++q)
            if (v[q] > bv) { bv = v[q]; bq = q; }
        int bi = (bv == -INFINITY) ? 0x7fffffff : lane + 32 * bq;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) {
#pragma unroll
            for (int q = 0; q < NQ; ++q)
                if (q == (bi >> 5)) v[q] = -INFINITY;  // taken
        }
        if (lane == j) { sel_i = bi; sel_v = bv; }
    }
    if (mode == MOE_ROUTER_SOFTMAX_TOPK) {
        const float p = (lane < K) ? __expf(sel_v - mx) / z : 0.0f;
        const float ps = warp_sum(p);
        w = (norm ? p / ps : p) * scale;
    } else {
        const float m0 = __shfl_sync(0xffffffffu, sel_v, 0);
        const float ex = (lane < K) ? __expf(sel_v - m0) : 0.0f;
        w = ex / warp_sum(ex);
    }
}

// The same for two tokens at once (two independent register sets, so the
// compiler interleaves their loads and compare chains).
template <int NQ>
__device__ __forceinline__ void warp_select2(const float *la, const float *lb, int E, int K, int mode, int norm,
                                             float scale, int lane, int (&sel_i)[2], float (&sel_v)[2],
                                             float (&w)[2])
{
    float v[2][NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const bool in = lane + 32 * q < E;
        v[0][q] = in ? __ldcg(la + lane + 32 * q) : -INFINITY;
        v[1][q] = in ? __ldcg(lb + lane + 32 * q) : -INFINITY;
    }
    float mx[2], z[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        mx[s] = -INFINITY;
#pragma unroll
        for (int q = 0; q < NQ; ++q) mx[s] = fmaxf(mx[s], v[s][q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int s = 0; s < 2; ++s) mx[s] = fmaxf(mx[s], __shfl_xor_sync(0xffffffffu, mx[s], o));
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        z[s] = 0.0f;
        if (mode == MOE_ROUTER_SOFTMAX_TOPK) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) z[s] += (lane + 32 * q < E) ? __expf(v[s][q] - mx[s]) : 0.0f;
        }
    }
    if (mode == MOE_ROUTER_SOFTMAX_TOPK) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int s = 0; s < 2; ++s) z[s] += __shfl_xor_sync(0xffffffffu, z[s], o);
    }
    sel_i[0] = sel_i[1] = -1;
    sel_v[0] = sel_v[1] = 0.0f;
    for (int j = 0; j < K; ++j) {
        float bv[2];
        int bi[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            bv[s] = v[s][0];
            int bq = 0;
#pragma unroll
            for (int q = 1; q < NQ; ++q)
                if (v[s][q] > bv[s]) { bv[s] = v[s][q]; bq = q; }
            bi[s] = (bv[s] == -INFINITY) ? 0x7fffffff : lane + 32 * bq;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv[s], o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi[s], o);
                if (ov > bv[s] || (ov == bv[s] && oi < bi[s])) { bv[s] = ov; bi[s] = oi; }
            }
        }
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if ((bi[s] & 31) == lane) {
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    if (q == (bi[s] >> 5)) v[s][q] = -INFINITY;  // taken
            }
            if (lane == j) { sel_i[s] = bi[s]; sel_v[s] = bv[s]; }
        }
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        if (mode == MOE_ROUTER_SOFTMAX_TOPK) {
            const float p = (lane < K) ? __expf(sel_v[s] - mx[s]) / z[s] : 0.0f;
            const float ps = warp_sum(p);
            w[s] = (norm ? p / ps : p) * scale;
        } else {
            const float m0 = __shfl_sync(0xffffffffu, sel_v[s], 0);
            const float ex = (lane < K) ? __expf(sel_v[s] - m0) : 0.0f;
            w[s] = ex / warp_sum(ex);
        }
    }
}

__device__ __forceinline__ void warp_select2_any(const float *la, const float *lb, int E, int K, int mode, int norm,
                                                 float scale, int lane, int (&sel_i)[2], float (&sel_v)[2],
                                                 float (&w)[2])
{
    const int nq = (E + 31) / 32;
    if (nq <= 1) warp_select2<1>(la, lb, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 2) warp_select2<2>(la, lb, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 4) warp_select2<4>(la, lb, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 8) warp_select2<8>(la, lb, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 16) warp_select2<16>(la, lb, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else warp_select2<32>(la, lb, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
}

// dispatch on the number of logits per lane (E <= 1024)
__device__ __forceinline__ void warp_select_any(const float *l, int E, int K, int mode, int norm, float scale, int lane,
                                                int &sel_i, float &sel_v, float &w)
{
    const int nq = (E + 31) / 32;
    if (nq <= 1) warp_select<1>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 2) warp_select<2>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 4) warp_select<4>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 8) warp_select<8>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else if (nq <= 16) warp_select<16>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    else warp_select<32>(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
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
int launch_select(const Layer &L, int T, cudaStream_t s);
int launch_group(const Layer &L, int T, bool build_tiles, cudaStream_t s);
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
void dectc_release(Layer &L);
// which: 0 = router logits, 1 = selection + gate/up + down (writes out)
int launch_dectc(const Layer &L, const void *x, int T, void *out, int which, cudaStream_t s);

// tensor-core path (expert_tc.cu)
bool tc_supported(const Layer &L, std::string &why);
int tc_prepare(Layer &L);  // tensor maps over the layer's weights/workspace; 0 on success
void tc_release(Layer &L);
// which: 0 = gather token rows, 1 = gate/up GEMM + activation, 2 = down GEMM + weight
int launch_experts_tc(const Layer &L, const void *x, int T, int which, cudaStream_t s);
void tc_tile_caps(const Layer &L, int &max_up, int &max_down);
int launch_tc_router(const Layer &L, const void *x, int T, cudaStream_t s);

constexpr int MAX_LAUNCHES_PER_FORWARD = 8;

// tile geometry of the tensor-core path (used by the grouping kernel)
constexpr int TC_BM = 128;       // token rows per tile
constexpr int TC_BN_UP = 128;    // gate/up tile: 64 gate + 64 up columns -> 64 h columns
constexpr int TC_BN_DOWN = 128;  // down tile: output columns
constexpr int TC_BK = 64;        // K elements per pipeline stage (128 bytes of bf16)

}  // namespace moe
