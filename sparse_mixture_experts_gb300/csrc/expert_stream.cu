// expert_stream.cu -- weight-streaming expert kernels (CUDA cores) and the
// fixed-order combine.
//
// Expert ("Llama Forward Pass", SwiGLU FFN and Mixture of Experts;
// "Phase 19: MoE -- gpt-oss-20b", section 2 Experts):
//   gate = W_gate,e x (+ b), up = W_up,e x (+ b), h = act(gate, up),
//   y = W_down,e h (+ b_down,e)
// Shared expert ("Qwen3.5-MoE Model Implementation", MoE routing): SwiGLU on
// every token, scaled by sigmoid(w_sh . x).
// Combine: out[t] = sum over slots in fixed order of w_slot * y_slot, then
// the shared slot; no floating-point atomics, so results are reproducible.
//
// The expert kernels walk "groups": the routed experts that received tokens
// (the grouping kernel lists them) and then the shared expert.  Each block
// streams a tile of one group's weight rows exactly once with 16-byte loads
// and applies it to every token routed to that group, so the weight bytes read
// are those of the selected experts only.  This path serves small token
// counts (decode) and every fp32 layer.
#include "moe_internal.cuh"

namespace moe {

struct StreamArgs {
    const void *x;
    int T, K, E, H, F, Fs, Fmax, Tmax;
    const int *counts, *offsets, *expert_rows, *active;
    const RouteMeta *meta;
    const void *gate_w, *up_w, *down_w;
    const float *gate_b, *up_b, *down_b;
    const void *sh_gate_w, *sh_up_w, *sh_down_w;
    const float *topk_w, *sh_gate;
    void *h;
    float *ys;         // [T][K+1][H] fp32
    float alpha, limit;
};

// Resolve grid row `g` to a group.  Returns false if the group is empty.
struct Group {
    int e;          // expert index, E for the shared expert
    int n;          // rows (tokens) in the group
    int row0;       // first row of the group in the activation buffer
    const int *pairs; // pair ids (t*K+slot) or nullptr for the shared expert (pair = token)
    int fd;         // ff width of the group
};

__device__ __forceinline__ bool resolve_group(const StreamArgs &a, int g, Group &G)
{
    const int n_active = a.meta->n_active;
    if (g < n_active) {
        G.e = a.active[g];
        G.n = a.counts[G.e];
        G.row0 = a.offsets[G.e];
        G.pairs = a.expert_rows + G.row0;
        G.fd = a.F;
        return G.n > 0;
    }
    if (g == n_active && a.Fs > 0) {
        G.e = a.E;
        G.n = a.T;
        G.row0 = a.T * a.K;
        G.pairs = nullptr;
        G.fd = a.Fs;
        return true;
    }
    return false;
}

constexpr int UP_ROWS = 16;   // ff rows (gate and up) per block
constexpr int DOWN_ROWS = 32; // hidden rows per block
constexpr int TOK = 8;        // tokens per pass

// ---------------------------------------------------------------------------
// gate/up + activation: h[row0 + j][f] = act(gate_f . x_j, up_f . x_j)
// ---------------------------------------------------------------------------
template <typename TW, int ACT>
__global__ void __launch_bounds__(256) expert_up_stream_kernel(StreamArgs a)
{
    constexpr int V = Vec<TW>::N;
    Group G;
    if (!resolve_group(a, blockIdx.y, G)) return;
    const int f0 = blockIdx.x * UP_ROWS;
    if (f0 >= G.fd) return;
    const bool shared = G.e == a.E;
    const TW *Wg = shared ? (const TW *)a.sh_gate_w : (const TW *)a.gate_w + (size_t)G.e * a.F * a.H;
    const TW *Wu = shared ? (const TW *)a.sh_up_w : (const TW *)a.up_w + (size_t)G.e * a.F * a.H;
    const float *bg = (!shared && a.gate_b) ? a.gate_b + (size_t)G.e * a.F : nullptr;
    const float *bu = (!shared && a.up_b) ? a.up_b + (size_t)G.e * a.F : nullptr;
    const TW *x = (const TW *)a.x;
    TW *h = (TW *)a.h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = a.H / V;

    for (int f = f0 + warp; f < min(f0 + UP_ROWS, G.fd); f += 8) {
        const TW *wg = Wg + (size_t)f * a.H;
        const TW *wu = Wu + (size_t)f * a.H;
        const float bgf = bg ? bg[f] : 0.0f, buf = bu ? bu[f] : 0.0f;
        for (int j0 = 0; j0 < G.n; j0 += TOK) {
            const int nt = min(TOK, G.n - j0);
            int tok[TOK];
#pragma unroll
            for (int j = 0; j < TOK; ++j) {
                int jj = j0 + min(j, nt - 1);
                tok[j] = G.pairs ? G.pairs[jj] / a.K : jj;
            }
            float ag[TOK], au[TOK];
#pragma unroll
            for (int j = 0; j < TOK; ++j) ag[j] = au[j] = 0.0f;
#pragma unroll 2
            for (int c = lane; c < nvec; c += 32) {
                Vec<TW> vg, vu;
                vg.load_stream(wg + (size_t)c * V);
                vu.load_stream(wu + (size_t)c * V);
#pragma unroll
                for (int j = 0; j < TOK; ++j) {
                    if (j < nt) {
                        Vec<TW> xv;
                        xv.load(x + (size_t)tok[j] * a.H + (size_t)c * V);
#pragma unroll
                        for (int q = 0; q < V; ++q) {
                            ag[j] = fmaf(vg.v[q], xv.v[q], ag[j]);
                            au[j] = fmaf(vu.v[q], xv.v[q], au[j]);
                        }
                    }
                }
            }
            float mine_g = 0.0f, mine_u = 0.0f;
#pragma unroll
            for (int j = 0; j < TOK; ++j) {
                float sg = warp_sum(ag[j]);
                float su = warp_sum(au[j]);
                if (lane == j) { mine_g = sg; mine_u = su; }
            }
            if (lane < nt) {
                float v = shared ? activation<MOE_ACT_SWIGLU>(mine_g, mine_u, a.alpha, a.limit)
                                 : activation<ACT>(mine_g + bgf, mine_u + buf, a.alpha, a.limit);
                store_out(h + (size_t)(G.row0 + j0 + lane) * a.Fmax + f, v);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// down + routing weight: ys[t][slot][i] = w * (down_i . h_j + b_i)
// ---------------------------------------------------------------------------
template <typename TW>
__global__ void __launch_bounds__(256) expert_down_stream_kernel(StreamArgs a)
{
    constexpr int V = Vec<TW>::N;
    constexpr int RW = 4;  // rows per warp pass
    Group G;
    if (!resolve_group(a, blockIdx.y, G)) return;
    const int i0 = blockIdx.x * DOWN_ROWS;
    if (i0 >= a.H) return;
    const bool shared = G.e == a.E;
    const int fd = G.fd;
    const TW *Wd = shared ? (const TW *)a.sh_down_w : (const TW *)a.down_w + (size_t)G.e * a.H * a.F;
    const float *bd = (!shared && a.down_b) ? a.down_b + (size_t)G.e * a.H : nullptr;
    const TW *h = (const TW *)a.h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = fd / V;
    const int S = a.K + 1;

    for (int ib = i0 + warp * RW; ib < min(i0 + DOWN_ROWS, a.H); ib += 8 * RW) {
        const int nr = min(RW, a.H - ib);
        for (int j0 = 0; j0 < G.n; j0 += TOK) {
            const int nt = min(TOK, G.n - j0);
            float acc[RW][TOK];
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int j = 0; j < TOK; ++j) acc[r][j] = 0.0f;
            for (int c = lane; c < nvec; c += 32) {
                Vec<TW> wv[RW];
#pragma unroll
                for (int r = 0; r < RW; ++r)
                    if (r < nr) wv[r].load_stream(Wd + (size_t)(ib + r) * fd + (size_t)c * V);
#pragma unroll
                for (int j = 0; j < TOK; ++j) {
                    if (j < nt) {
                        Vec<TW> hv;
                        hv.load(h + (size_t)(G.row0 + j0 + j) * a.Fmax + (size_t)c * V);
#pragma unroll
                        for (int r = 0; r < RW; ++r)
                            if (r < nr)
#pragma unroll
                                for (int q = 0; q < V; ++q) acc[r][j] = fmaf(wv[r].v[q], hv.v[q], acc[r][j]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                float mine = 0.0f;
#pragma unroll
                for (int j = 0; j < TOK; ++j) {
                    float s = warp_sum(acc[r][j]);
                    if (lane == j) mine = s;
                }
                if (r < nr && lane < nt) {
                    const int row = ib + r;
                    const int j = j0 + lane;
                    int t, slot;
                    float wgt;
                    if (shared) { t = j; slot = a.K; wgt = a.sh_gate[t]; }
                    else {
                        const int p = G.pairs[j];
                        t = p / a.K; slot = p - t * a.K; wgt = a.topk_w[p];
                    }
                    const float y = mine + (bd ? bd[row] : 0.0f);
                    a.ys[((size_t)t * S + slot) * a.H + row] = wgt * y;
                }
            }
        }
    }
}

static StreamArgs make_args(const Layer &L, const void *x, int T)
{
    StreamArgs a;
    a.x = x;
    a.T = T; a.K = L.K; a.E = L.E; a.H = L.H; a.F = L.F; a.Fs = L.Fs; a.Fmax = L.Fmax; a.Tmax = L.Tmax;
    a.counts = L.counts; a.offsets = L.offsets; a.expert_rows = L.expert_rows; a.active = L.active;
    a.meta = L.meta;
    a.gate_w = L.gate_w; a.up_w = L.up_w; a.down_w = L.down_w;
    a.gate_b = L.gate_b; a.up_b = L.up_b; a.down_b = L.down_b;
    a.sh_gate_w = L.sh_gate_w; a.sh_up_w = L.sh_up_w; a.sh_down_w = L.sh_down_w;
    a.topk_w = L.topk_w; a.sh_gate = L.sh_gate;
    a.h = L.h; a.ys = L.ys;
    a.alpha = L.cfg.act_alpha; a.limit = L.cfg.act_limit;
    return a;
}

int launch_experts_stream(const Layer &L, const void *x, int T, int which, cudaStream_t s)
{
    StreamArgs a = make_args(L, x, T);
    // at most min(E, T*K) experts receive tokens, plus the shared expert
    const int groups = min(L.E, T * L.K) + (L.Fs > 0 ? 1 : 0);
    const bool bf = L.cfg.w_dtype == MOE_DT_BF16;
    const bool clamp = L.cfg.act == MOE_ACT_CLAMP_GLU;
    if (which == 0) {
        dim3 gu((L.Fmax + UP_ROWS - 1) / UP_ROWS, groups);
        if (bf) {
            if (clamp) expert_up_stream_kernel<__nv_bfloat16, MOE_ACT_CLAMP_GLU><<<gu, 256, 0, s>>>(a);
            else expert_up_stream_kernel<__nv_bfloat16, MOE_ACT_SWIGLU><<<gu, 256, 0, s>>>(a);
        } else {
            if (clamp) expert_up_stream_kernel<float, MOE_ACT_CLAMP_GLU><<<gu, 256, 0, s>>>(a);
            else expert_up_stream_kernel<float, MOE_ACT_SWIGLU><<<gu, 256, 0, s>>>(a);
        }
    } else {
        dim3 gd((L.H + DOWN_ROWS - 1) / DOWN_ROWS, groups);
        if (bf) expert_down_stream_kernel<__nv_bfloat16><<<gd, 256, 0, s>>>(a);
        else expert_down_stream_kernel<float><<<gd, 256, 0, s>>>(a);
    }
    return 1;
}

// ---------------------------------------------------------------------------
// combine: out[t][i] = sum_{slot < K} ys[t][slot][i] (+ ys[t][K][i]); ys holds the
// weighted per-slot outputs in fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 load4_stream(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }

template <typename TO>
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ ys, int T, int K, int H, int has_shared,
                                                      TO *__restrict__ out)
{
    const int S = K + 1;
    const int nslots = K + (has_shared ? 1 : 0);
    const size_t n4 = (size_t)T * H / 4;
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += (size_t)gridDim.x * blockDim.x) {
        const size_t e = q * 4;
        const size_t t = e / H, i = e - t * H;
        const float *p = ys + t * S * H + i;
        float4 acc = load4_stream(p);
        for (int sl = 1; sl < nslots; ++sl) {
            const float4 v = load4_stream(p + (size_t)sl * H);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        TO *o = out + e;
        store_out(o + 0, acc.x);
        store_out(o + 1, acc.y);
        store_out(o + 2, acc.z);
        store_out(o + 3, acc.w);
    }
}

int launch_combine(const Layer &L, int T, void *out, cudaStream_t s)
{
    const size_t n4 = (size_t)T * L.H / 4;
    size_t want = (n4 + 255) / 256, cap = (size_t)L.num_sms * 8;
    int blocks = (int)(want < cap ? want : cap);
    blocks = max(blocks, 1);
    const int hs = L.Fs > 0;
    if (L.cfg.out_dtype == MOE_DT_BF16) combine_kernel<<<blocks, 256, 0, s>>>(L.ys, T, L.K, L.H, hs, (__nv_bfloat16 *)out);
    else combine_kernel<<<blocks, 256, 0, s>>>(L.ys, T, L.K, L.H, hs, (float *)out);
    return 1;
}

}  // namespace moe
