// decode.cu -- the whole MoE layer in one cooperative kernel, for small token
// counts (decode batches), where the time is the HBM stream of the selected
// experts' weights and kernel boundaries would dominate.
//
// Phase A (all blocks, warp jobs): router logits l[t][e] = Wr[e].x[t] (+ b)
//   and the shared-expert gate/up rows, h_sh[t][f] = silu(g).u, which do not
//   depend on the routing ("Qwen3.5-MoE Model Implementation", MoE routing:
//   router, shared expert with scalar sigmoid gate).
// -- grid barrier --
// Phase B: every block selects the top-k of every token from the logits
//   (same code and inputs in every block, so the same result) -- softmax ->
//   top-k -> renormalise -> scale, or top-k -> softmax for the gpt-oss form --
//   lists the experts that received tokens, prefetches into L2 the down rows
//   it will need in phase C, then computes the routed gate/up rows:
//   h[t*k + j][f] = act(gate_f.x_t (+b), up_f.x_t (+b)) for each selected e.
//   ("Llama Forward Pass", Mixture of Experts; "Phase 19: MoE --
//   gpt-oss-20b", section 2 Router and Experts)
// -- grid barrier --
// Phase C: per tile of output rows, y = W_down,e h (+ b_down) for every
//   (token, slot) and the shared expert, then
//   out[t][i] = sum_{j<k} w[t][j] y[t][j][i] + sigmoid(l_sh[t]) y_sh[t][i],
//   summed in slot order (deterministic), written straight to `out`.
//
// Each weight row is read once per forward with 16-byte loads; the grid
// barriers spin with a bound (a second by default) and, on timeout, record an
// error and end the kernel.
#include "moe_internal.cuh"

namespace moe {

constexpr int DEC_THREADS = 256;
constexpr int DEC_WARPS = DEC_THREADS / 32;
constexpr int DEC_TMAX = 8;       // tokens
constexpr int DEC_PAIRS = 256;    // max tokens * top_k
constexpr int DEC_FR = 16;        // ff rows per phase-B item
constexpr int DEC_RC_MAX = 16;    // output rows per phase-C item

struct DecodeArgs {
    const void *x;
    void *out;
    int T, K, E, H, F, Fs, R, Fmax;
    int mode, norm, out_bf16;
    float scale, alpha, limit;
    const void *router_w;
    const float *router_b;
    const void *gate_w, *up_w, *down_w;
    const float *gate_b, *up_b, *down_b;
    const void *sh_gate_w, *sh_up_w, *sh_down_w;
    float *logits;
    int *topk_idx;
    float *topk_w;
    float *sh_gate;
    int *counts;
    void *h;
    unsigned *gbar;  // [0] arrivals, [1] generation
    int *status;
    unsigned long long wait_ns;  // bound of a grid-barrier wait
    int inject;                  // test-only: barriers that never complete
    int rc;           // output rows per phase-C item
    int prefetch;     // prefetch phase-C rows into L2 during phase B
};

__device__ __forceinline__ unsigned long long dec_timer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Grid-wide barrier for a cooperative launch; the spin is bounded by wait_ns.
// Returns false (in every thread of the block) when the wait ran out: the
// error is recorded and the caller returns, since other blocks' results are
// not all there.  `extra` (test-only fault injection) raises the arrival
// count the last block must see, so that no block ever completes the barrier.
__device__ __forceinline__ bool grid_barrier(unsigned *gbar, int *status, unsigned long long wait_ns, int extra)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        volatile unsigned *gen = gbar + 1;
        const unsigned g = *gen;
        __threadfence();
        const unsigned arrived = atomicAdd(gbar, 1u);
        if (arrived == gridDim.x - 1 + (unsigned)extra) {
            gbar[0] = 0;
            __threadfence();
            atomicExch(gbar + 1, g + 1);
        } else {
            const unsigned long long t0 = dec_timer();
            unsigned it = 0;
            while (*gen == g) {
                if ((++it & 63) == 0 && dec_timer() - t0 > wait_ns) {
                    record_error(status, DEV_TIMEOUT_GRID_BARRIER);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    // bulk prefetch: 16-byte aligned address, size a multiple of 16
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <typename TW> __device__ __forceinline__ void ld_cg(Vec<TW> &v, const TW *p);
template <> __device__ __forceinline__ void ld_cg<__nv_bfloat16>(Vec<__nv_bfloat16> &v, const __nv_bfloat16 *p)
{
    v.unpack(__ldcg(reinterpret_cast<const uint4 *>(p)));
}
template <> __device__ __forceinline__ void ld_cg<float>(Vec<float> &v, const float *p)
{
    float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
    v.v[0] = a.x; v.v[1] = a.y; v.v[2] = a.z; v.v[3] = a.w;
}

// warp: acc[t] (lane partials) += row . x[tok[t]] for t < n; x rows of H
template <typename TW>
__device__ __forceinline__ void warp_row_dot(const TW *__restrict__ row, const TW *__restrict__ x, const int *tok,
                                             int n, int H, int lane, float (&acc)[DEC_TMAX])
{
    constexpr int V = Vec<TW>::N;
    const int nvec = H / V;
#pragma unroll 4
    for (int c = lane; c < nvec; c += 32) {
        Vec<TW> w;
        w.load_stream(row + (size_t)c * V);
#pragma unroll
        for (int t = 0; t < DEC_TMAX; ++t) {
            if (t < n) {
                Vec<TW> xv;
                xv.load(x + (size_t)tok[t] * H + (size_t)c * V);
#pragma unroll
                for (int q = 0; q < V; ++q) acc[t] = fmaf(w.v[q], xv.v[q], acc[t]);
            }
        }
    }
}

// warp: gate and up rows at once
template <typename TW>
__device__ __forceinline__ void warp_pair_dot(const TW *__restrict__ g_row, const TW *__restrict__ u_row,
                                              const TW *__restrict__ x, const int *tok, int n, int H, int lane,
                                              float (&ag)[DEC_TMAX], float (&au)[DEC_TMAX])
{
    constexpr int V = Vec<TW>::N;
    const int nvec = H / V;
#pragma unroll 4
    for (int c = lane; c < nvec; c += 32) {
        Vec<TW> wg, wu;
        wg.load_stream(g_row + (size_t)c * V);
        wu.load_stream(u_row + (size_t)c * V);
#pragma unroll
        for (int t = 0; t < DEC_TMAX; ++t) {
            if (t < n) {
                Vec<TW> xv;
                xv.load(x + (size_t)tok[t] * H + (size_t)c * V);
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    ag[t] = fmaf(wg.v[q], xv.v[q], ag[t]);
                    au[t] = fmaf(wu.v[q], xv.v[q], au[t]);
                }
            }
        }
    }
}

// (value, index) ordering: larger value first, lower index on equal values
__device__ __forceinline__ bool dec_better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

template <typename TW, int ACT>
__global__ void __launch_bounds__(DEC_THREADS, 2) moe_decode_kernel(const DecodeArgs a)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const TW *x = (const TW *)a.x;
    TW *h = (TW *)a.h;
    const int T = a.T, K = a.K, E = a.E, H = a.H, F = a.F, Fs = a.Fs, R = a.R;
    const int P = T * K;

    __shared__ int s_idx[DEC_PAIRS];
    __shared__ float s_w[DEC_PAIRS];
    __shared__ float s_gsh[DEC_TMAX];
    __shared__ int s_cnt[1024];
    __shared__ int s_act[DEC_PAIRS];          // active experts, ascending
    __shared__ unsigned char s_list[DEC_PAIRS][DEC_TMAX];  // pair ids of each active expert
    __shared__ unsigned char s_nlist[DEC_PAIRS];
    __shared__ int s_nact;
    __shared__ float s_y[DEC_PAIRS + DEC_TMAX][DEC_RC_MAX];

    int tok_all[DEC_TMAX];
#pragma unroll
    for (int t = 0; t < DEC_TMAX; ++t) tok_all[t] = t < T ? t : 0;

    // ------------------------------ phase A ------------------------------
    {
        const int gw = blockIdx.x * DEC_WARPS + warp, nw = G * DEC_WARPS;
        const int jobs = R + Fs;
        for (int j = gw; j < jobs; j += nw) {
            if (j < R) {
                float acc[DEC_TMAX];
#pragma unroll
                for (int t = 0; t < DEC_TMAX; ++t) acc[t] = 0.0f;
                warp_row_dot<TW>((const TW *)a.router_w + (size_t)j * H, x, tok_all, T, H, lane, acc);
                const float b = (a.router_b && j < E) ? a.router_b[j] : 0.0f;
#pragma unroll
                for (int t = 0; t < DEC_TMAX; ++t) {
                    if (t < T) {
                        float s = warp_sum(acc[t]);
                        if (lane == 0) a.logits[(size_t)t * R + j] = s + b;
                    }
                }
            } else {
                const int f = j - R;
                float ag[DEC_TMAX], au[DEC_TMAX];
#pragma unroll
                for (int t = 0; t < DEC_TMAX; ++t) ag[t] = au[t] = 0.0f;
                warp_pair_dot<TW>((const TW *)a.sh_gate_w + (size_t)f * H, (const TW *)a.sh_up_w + (size_t)f * H, x,
                                  tok_all, T, H, lane, ag, au);
#pragma unroll
                for (int t = 0; t < DEC_TMAX; ++t) {
                    if (t < T) {
                        float g = warp_sum(ag[t]), u = warp_sum(au[t]);
                        if (lane == 0)
                            store_out(h + (size_t)(P + t) * a.Fmax + f, activation<MOE_ACT_SWIGLU>(g, u, 0.f, 0.f));
                    }
                }
            }
        }
        // the shared expert's down rows of this block's phase-C items
        if (a.prefetch && Fs > 0 && threadIdx.x == 0) {
            for (int i = blockIdx.x; i * a.rc < H; i += G) {
                const int r0 = i * a.rc, nr = min(a.rc, H - r0);
                prefetch_l2((const TW *)a.sh_down_w + (size_t)r0 * Fs, (uint32_t)(nr * Fs * sizeof(TW)));
            }
        }
    }
    if (!grid_barrier(a.gbar, a.status, a.wait_ns, a.inject)) return;

    // ------------------------------ phase B ------------------------------
    for (int t = warp; t < T; t += DEC_WARPS) {
        const float *l = a.logits + (size_t)t * R;
        float mx = -INFINITY;
        for (int e = lane; e < E; e += 32) mx = fmaxf(mx, __ldcg(l + e));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int sel_i = -1;
        float sel_v = 0.0f;
        unsigned taken = 0;
        for (int j = 0; j < K; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            int q = 0;
            for (int e = lane; e < E; e += 32, ++q) {
                if (taken & (1u << q)) continue;
                float v = __ldcg(l + e);
                if (bi == 0x7fffffff || dec_better(v, e, bv, bi)) { bv = v; bi = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi != 0x7fffffff && (bi == 0x7fffffff || dec_better(ov, oi, bv, bi))) { bv = ov; bi = oi; }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) { sel_i = bi; sel_v = bv; }
        }
        float w;
        if (a.mode == MOE_ROUTER_SOFTMAX_TOPK) {
            float z = 0.0f;
            for (int e = lane; e < E; e += 32) z += __expf(__ldcg(l + e) - mx);
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
        if (lane == 0) s_gsh[t] = Fs > 0 ? 1.0f / (1.0f + __expf(-__ldcg(l + E))) : 0.0f;
    }
    for (int e = threadIdx.x; e < E; e += DEC_THREADS) s_cnt[e] = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += DEC_THREADS) atomicAdd(&s_cnt[s_idx[p]], 1);
    __syncthreads();
    {
        // experts that received tokens, ascending: ballot compaction, DEC_THREADS experts per round
        __shared__ int s_wtot[DEC_WARPS];
        int base = 0;
        for (int e0 = 0; e0 < E; e0 += DEC_THREADS) {
            const int e = e0 + threadIdx.x;
            const bool on = e < E && s_cnt[e] > 0;
            const unsigned m = __ballot_sync(0xffffffffu, on);
            if (lane == 0) s_wtot[warp] = __popc(m);
            __syncthreads();
            int before = 0, all = 0;
#pragma unroll
            for (int w = 0; w < DEC_WARPS; ++w) {
                before += w < warp ? s_wtot[w] : 0;
                all += s_wtot[w];
            }
            if (on) s_act[base + before + __popc(m & ((1u << lane) - 1u))] = e;
            base += all;
            __syncthreads();
        }
        if (threadIdx.x == 0) s_nact = base;
    }
    __syncthreads();
    const int n_act = s_nact;
    for (int ai = threadIdx.x; ai < n_act; ai += DEC_THREADS) {
        const int e = s_act[ai];
        int n = 0;
        for (int p = 0; p < P; ++p)
            if (s_idx[p] == e) s_list[ai][n++] = (unsigned char)p;
        s_nlist[ai] = (unsigned char)n;
    }
    if (blockIdx.x == 0) {
        for (int p = threadIdx.x; p < P; p += DEC_THREADS) {
            a.topk_idx[p] = s_idx[p];
            a.topk_w[p] = s_w[p];
        }
        for (int t = threadIdx.x; t < T; t += DEC_THREADS)
            if (Fs > 0) a.sh_gate[t] = s_gsh[t];
        for (int e = threadIdx.x; e < E; e += DEC_THREADS) a.counts[e] = s_cnt[e];
    }
    __syncthreads();

    // L2 prefetch of the routed down rows this block reads in phase C
    if (a.prefetch) {
        const int n_items_c = (H + a.rc - 1) / a.rc;
        const int per_item = n_act;
        for (int q = threadIdx.x; q < per_item * ((n_items_c - blockIdx.x + G - 1) / G); q += DEC_THREADS) {
            const int i = blockIdx.x + (q / per_item) * G;
            const int e = s_act[q % per_item];
            const int r0 = i * a.rc, nr = min(a.rc, H - r0);
            prefetch_l2((const TW *)a.down_w + ((size_t)e * H + r0) * F, (uint32_t)(nr * F * sizeof(TW)));
        }
    }

    // routed gate/up: item = (active expert, tile of DEC_FR ff rows)
    {
        const int tiles_per_e = F / DEC_FR;
        const int n_items = n_act * tiles_per_e;
        for (int i = blockIdx.x; i < n_items; i += G) {
            const int ai = i / tiles_per_e, ft = i - ai * tiles_per_e;
            const int e = s_act[ai];
            const int n = s_nlist[ai];
            int tok[DEC_TMAX];
#pragma unroll
            for (int t = 0; t < DEC_TMAX; ++t) tok[t] = s_list[ai][t < n ? t : 0] / K;
            const TW *Wg = (const TW *)a.gate_w + (size_t)e * F * H;
            const TW *Wu = (const TW *)a.up_w + (size_t)e * F * H;
            for (int f = ft * DEC_FR + warp; f < (ft + 1) * DEC_FR; f += DEC_WARPS) {
                float ag[DEC_TMAX], au[DEC_TMAX];
#pragma unroll
                for (int t = 0; t < DEC_TMAX; ++t) ag[t] = au[t] = 0.0f;
                warp_pair_dot<TW>(Wg + (size_t)f * H, Wu + (size_t)f * H, x, tok, n, H, lane, ag, au);
                const float bg = a.gate_b ? a.gate_b[(size_t)e * F + f] : 0.0f;
                const float bu = a.up_b ? a.up_b[(size_t)e * F + f] : 0.0f;
#pragma unroll
                for (int t = 0; t < DEC_TMAX; ++t) {
                    if (t < n) {
                        float g = warp_sum(ag[t]), u = warp_sum(au[t]);
                        if (lane == 0)
                            store_out(h + (size_t)s_list[ai][t] * a.Fmax + f,
                                      activation<ACT>(g + bg, u + bu, a.alpha, a.limit));
                    }
                }
            }
        }
    }
    if (!grid_barrier(a.gbar, a.status, a.wait_ns, a.inject)) return;

    // ------------------------------ phase C ------------------------------
    {
        constexpr int V = Vec<TW>::N;
        const int n_items = (H + a.rc - 1) / a.rc;
        const int n_groups = n_act + (Fs > 0 ? 1 : 0);
        for (int i = blockIdx.x; i < n_items; i += G) {
            const int r0 = i * a.rc, nr = min(a.rc, H - r0);
            // warps over (group, 4 rows): y of every (token, slot) of the group
            const int nquads = (nr + 3) / 4;
            for (int job = warp; job < n_groups * nquads; job += DEC_WARPS) {
                const int gi = job / nquads, rr0 = (job - gi * nquads) * 4;
                const int nrr = min(4, nr - rr0);
                const bool shared = gi == n_act;
                const int fd = shared ? Fs : F;
                const TW *w0 = shared ? (const TW *)a.sh_down_w + (size_t)(r0 + rr0) * Fs
                                      : (const TW *)a.down_w + ((size_t)s_act[gi] * H + r0 + rr0) * F;
                const int n = shared ? T : s_nlist[gi];
                int hrow[DEC_TMAX];
#pragma unroll
                for (int t = 0; t < DEC_TMAX; ++t) hrow[t] = shared ? P + (t < n ? t : 0) : s_list[gi][t < n ? t : 0];
                float acc[4][DEC_TMAX];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int t = 0; t < DEC_TMAX; ++t) acc[r][t] = 0.0f;
                const int nvec = fd / V;
#pragma unroll 2
                for (int c = lane; c < nvec; c += 32) {
                    Vec<TW> wv[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        if (r < nrr) wv[r].load_stream(w0 + (size_t)r * fd + (size_t)c * V);
#pragma unroll
                    for (int t = 0; t < DEC_TMAX; ++t) {
                        if (t < n) {
                            Vec<TW> hv;
                            ld_cg<TW>(hv, h + (size_t)hrow[t] * a.Fmax + (size_t)c * V);
#pragma unroll
                            for (int r = 0; r < 4; ++r)
                                if (r < nrr)
#pragma unroll
                                    for (int q = 0; q < V; ++q) acc[r][t] = fmaf(wv[r].v[q], hv.v[q], acc[r][t]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r < nrr) {
                        const float b = (!shared && a.down_b) ? a.down_b[(size_t)s_act[gi] * H + r0 + rr0 + r] : 0.0f;
#pragma unroll
                        for (int t = 0; t < DEC_TMAX; ++t) {
                            if (t < n) {
                                float sum = warp_sum(acc[r][t]);
                                if (lane == 0) s_y[hrow[t]][rr0 + r] = sum + b;
                            }
                        }
                    }
                }
            }
            __syncthreads();
            for (int q = threadIdx.x; q < T * nr; q += DEC_THREADS) {
                const int t = q / nr, rr = q - t * nr;
                float o = 0.0f;
                for (int j = 0; j < K; ++j) o += s_w[t * K + j] * s_y[t * K + j][rr];
                if (Fs > 0) o += s_gsh[t] * s_y[P + t][rr];
                const size_t oi = (size_t)t * H + r0 + rr;
                if (a.out_bf16) store_out((__nv_bfloat16 *)a.out + oi, o);
                else store_out((float *)a.out + oi, o);
            }
            __syncthreads();
        }
    }
}

bool decode_supported(const Layer &L, int T)
{
    return T >= 1 && T <= DEC_TMAX && T * L.K <= DEC_PAIRS && L.F % DEC_FR == 0 && L.decode_grid > 0;
}

int decode_prepare(Layer &L)
{
    auto occ = [&](const void *fn) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, DEC_THREADS, 0) != cudaSuccess) return 0;
        return nb;
    };
    int nb;
    if (L.cfg.w_dtype == MOE_DT_BF16)
        nb = L.cfg.act == MOE_ACT_CLAMP_GLU ? occ((const void *)moe_decode_kernel<__nv_bfloat16, MOE_ACT_CLAMP_GLU>)
                                            : occ((const void *)moe_decode_kernel<__nv_bfloat16, MOE_ACT_SWIGLU>);
    else
        nb = L.cfg.act == MOE_ACT_CLAMP_GLU ? occ((const void *)moe_decode_kernel<float, MOE_ACT_CLAMP_GLU>)
                                            : occ((const void *)moe_decode_kernel<float, MOE_ACT_SWIGLU>);
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, L.device);
    L.decode_grid = (coop && nb > 0) ? L.num_sms * (nb < 2 ? nb : 2) : 0;
    return 0;
}

int launch_decode(const Layer &L, const void *x, int T, void *out, cudaStream_t s)
{
    DecodeArgs a;
    a.x = x; a.out = out;
    a.T = T; a.K = L.K; a.E = L.E; a.H = L.H; a.F = L.F; a.Fs = L.Fs; a.R = L.R; a.Fmax = L.Fmax;
    a.mode = L.cfg.router_mode; a.norm = L.cfg.norm_topk_prob; a.out_bf16 = L.cfg.out_dtype == MOE_DT_BF16;
    a.scale = L.cfg.weights_scale; a.alpha = L.cfg.act_alpha; a.limit = L.cfg.act_limit;
    a.router_w = L.router_w; a.router_b = L.router_b;
    a.gate_w = L.gate_w; a.up_w = L.up_w; a.down_w = L.down_w;
    a.gate_b = L.gate_b; a.up_b = L.up_b; a.down_b = L.down_b;
    a.sh_gate_w = L.sh_gate_w; a.sh_up_w = L.sh_up_w; a.sh_down_w = L.sh_down_w;
    a.logits = L.logits; a.topk_idx = L.topk_idx; a.topk_w = L.topk_w; a.sh_gate = L.sh_gate; a.counts = L.counts;
    a.h = L.h;
    a.gbar = L.gbar;
    a.wait_ns = L.wait_ns;
    a.inject = L.inject;
    a.status = L.status;
    const int G = L.decode_grid;
    int rc = (L.H + G - 1) / G;
    a.rc = rc < 1 ? 1 : (rc > DEC_RC_MAX ? DEC_RC_MAX : rc);
    // prefetch the phase-C rows while they fit comfortably in L2
    const size_t down_bytes = (size_t)(T * L.K < L.E ? T * L.K : L.E) * L.H * L.F * L.wbytes;
    a.prefetch = down_bytes <= (size_t)48 << 20;
    void *args[] = {&a};
    const void *fn;
    if (L.cfg.w_dtype == MOE_DT_BF16)
        fn = L.cfg.act == MOE_ACT_CLAMP_GLU ? (const void *)moe_decode_kernel<__nv_bfloat16, MOE_ACT_CLAMP_GLU>
                                            : (const void *)moe_decode_kernel<__nv_bfloat16, MOE_ACT_SWIGLU>;
    else
        fn = L.cfg.act == MOE_ACT_CLAMP_GLU ? (const void *)moe_decode_kernel<float, MOE_ACT_CLAMP_GLU>
                                            : (const void *)moe_decode_kernel<float, MOE_ACT_SWIGLU>;
    if (cudaLaunchCooperativeKernel(fn, dim3(G), dim3(DEC_THREADS), args, 0, s) != cudaSuccess) return -1;
    return 1;
}

}  // namespace moe
