// route.cu -- router logits, expert selection and token grouping.
//
// Router ("Qwen3.5-MoE Model Implementation", MoE routing; "Phase 19: MoE --
// gpt-oss-20b", section 2 Router; "Llama Forward Pass", Mixture of Experts):
//   l[t][e] = sum_i Wr[e][i] x[t][i] (+ b[e]);  with a shared expert the
//   scalar-gate vector is router row E, so l[t][E] = w_sh . x[t].
// Selection, per token:
//   softmax form : p = softmax(l[0..E)), top-k, w = p_sel / sum p_sel
//                  (norm_topk_prob), w *= weights_scale
//   gpt-oss form : top-k on l (bias included), w = softmax over the k
//   ties go to the lower expert index; output order is descending weight.
// Grouping ("Engine", Prefill: tokens grouped by expert, gathered, projected,
// scattered back): for each expert the (token, slot) pairs routed to it in
// ascending token order, their count, the exclusive prefix sum of the counts
// (the expert's first row in the expert-sorted activation buffer), the list
// of experts that received tokens, and the tile lists of the tensor-core path.
// Everything is integer work with a fixed order, so it is deterministic.
#include "moe_internal.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// router logits: one warp per router row, tokens in chunks of 8; the row is
// re-read per chunk (from L2 after the first).
// ---------------------------------------------------------------------------
template <typename TW>
__global__ void __launch_bounds__(128) router_kernel(const TW *__restrict__ W, const float *__restrict__ bias,
                                                     const TW *__restrict__ x, int T, int H, int E, int R,
                                                     int tok_per_block, float *__restrict__ logits)
{
    constexpr int V = Vec<TW>::N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 4 + warp;
    if (r >= R) return;
    const int tbeg = blockIdx.y * tok_per_block;
    const int tend = min(T, tbeg + tok_per_block);
    const TW *w = W + (size_t)r * H;
    const int nvec = H / V;
    const float b = (bias != nullptr && r < E) ? bias[r] : 0.0f;
    for (int t0 = tbeg; t0 < tend; t0 += 8) {
        const int nt = min(8, tend - t0);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int c = lane; c < nvec; c += 32) {
            Vec<TW> wv;
            wv.load(w + (size_t)c * V);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j < nt) {
                    Vec<TW> xv;
                    xv.load(x + (size_t)(t0 + j) * H + (size_t)c * V);
#pragma unroll
                    for (int q = 0; q < V; ++q) acc[j] = fmaf(wv.v[q], xv.v[q], acc[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = warp_sum(acc[j]);
        if (lane < nt) {
            float v = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (lane == j) v = acc[j];
            logits[(size_t)(t0 + lane) * R + r] = v + b;
        }
    }
}

int launch_router(const Layer &L, const void *x, int T, cudaStream_t s)
{
    // spread tokens so that the grid covers the GPU for large T
    int row_blocks = (L.R + 3) / 4;
    int tok_per_block = T;
    if ((long long)row_blocks * 2 < 4LL * L.num_sms) {
        int want_y = (4 * L.num_sms + row_blocks - 1) / row_blocks;
        tok_per_block = max(8, (T + want_y - 1) / want_y);
        tok_per_block = (tok_per_block + 7) / 8 * 8;
    }
    dim3 grid(row_blocks, (T + tok_per_block - 1) / tok_per_block);
    if (L.cfg.w_dtype == MOE_DT_BF16)
        router_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>((const __nv_bfloat16 *)L.router_w, L.router_b,
                                                          (const __nv_bfloat16 *)x, T, L.H, L.E, L.R,
                                                          tok_per_block, L.logits);
    else
        router_kernel<float><<<grid, 128, 0, s>>>((const float *)L.router_w, L.router_b, (const float *)x, T, L.H,
                                                  L.E, L.R, tok_per_block, L.logits);
    return 1;
}

// ---------------------------------------------------------------------------
// selection: one warp per token
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) select_kernel(const float *__restrict__ logits, int T, int E, int R, int K,
                                                     int mode, int norm, float scale, int has_shared,
                                                     int *__restrict__ topk_idx, float *__restrict__ topk_w,
                                                     float *__restrict__ sh_gate)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    const float *l = logits + (size_t)t * R;
    int sel_i;
    float sel_v, w;
    warp_select_any(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    if (lane < K) {
        topk_idx[(size_t)t * K + lane] = sel_i;
        topk_w[(size_t)t * K + lane] = w;
    }
    if (has_shared && lane == 0) sh_gate[t] = 1.0f / (1.0f + __expf(-l[E]));
}

int launch_select(const Layer &L, int T, cudaStream_t s)
{
    const moe_config &c = L.cfg;
    select_kernel<<<(T + 7) / 8, 256, 0, s>>>(L.logits, T, L.E, L.R, L.K, c.router_mode, c.norm_topk_prob,
                                              c.weights_scale, L.Fs > 0, L.topk_idx, L.topk_w, L.sh_gate);
    return 1;
}

// ---------------------------------------------------------------------------
// grouping: one block per expert, the last block to finish finalises
// ---------------------------------------------------------------------------
constexpr int GT = 256;  // threads per grouping block

// exclusive prefix sum over the block's threads; *total gets the sum
__device__ int block_exclusive_scan(int v, int *total)
{
    __shared__ int warp_tot[GT / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < GT / 32; ++w) {
        int x = warp_tot[w];
        before += (w < warp) ? x : 0;
        all += x;
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

struct GroupArgs {
    const int *topk_idx;
    int T, K, E, Tmax;
    int has_shared, F, Fs, H;
    int *expert_rows, *counts, *offsets, *active;
    RouteMeta *meta;
    int build_tiles;
    TileDesc *up_tiles, *down_tiles;
    int max_up, max_down;
    int *status;
};

__global__ void __launch_bounds__(GT) group_kernel(GroupArgs a)
{
    const int e = blockIdx.x;
    __shared__ int s_base;
    __shared__ int s_last;
    if (threadIdx.x == 0) s_base = 0;
    __syncthreads();

    // pairs routed to expert e, in ascending token order (stable compaction)
    for (int t0 = 0; t0 < a.T; t0 += GT) {
        const int t = t0 + threadIdx.x;
        int slot = -1;
        if (t < a.T)
            for (int q = 0; q < a.K; ++q)
                if (__ldg(&a.topk_idx[(size_t)t * a.K + q]) == e) slot = q;
        int total;
        int pos = block_exclusive_scan(slot >= 0 ? 1 : 0, &total);
        if (slot >= 0) a.expert_rows[(size_t)e * a.Tmax + s_base + pos] = t * a.K + slot;
        __syncthreads();
        if (threadIdx.x == 0) s_base += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.counts[e] = s_base;
        __threadfence();
        int arrived = atomicAdd(&a.meta->ticket, 1);
        s_last = (arrived == a.E - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last block: prefix sums, active list, tile lists ----
    __shared__ int s_cnt[1024];
    __shared__ int s_act[1024];
    __shared__ int s_nact;
    for (int i = threadIdx.x; i < a.E; i += GT) s_cnt[i] = __ldcg(&a.counts[i]);
    __syncthreads();

    // each thread owns a contiguous run of up to 4 experts (E <= 1024)
    const int per = (a.E + GT - 1) / GT;
    const int beg = min(a.E, threadIdx.x * per), end = min(a.E, beg + per);
    int run = 0, run_act = 0;
    for (int i = beg; i < end; ++i) { run += s_cnt[i]; run_act += s_cnt[i] > 0; }
    int tot, tot_act;
    int off = block_exclusive_scan(run, &tot);
    int aoff = block_exclusive_scan(run_act, &tot_act);
    for (int i = beg; i < end; ++i) {
        a.offsets[i] = off;
        off += s_cnt[i];
        if (s_cnt[i] > 0) { s_act[aoff] = i; a.active[aoff] = i; ++aoff; }
    }
    if (threadIdx.x == 0) {
        a.offsets[a.E] = tot;
        s_nact = tot_act;
    }
    __syncthreads();

    int n_up = 0, n_down = 0;
    if (a.build_tiles) {
        // groups: active experts, then the shared expert
        const int n_groups = s_nact + (a.has_shared ? 1 : 0);
        const int n_dn = (a.H + TC_BN_DOWN - 1) / TC_BN_DOWN;
        int cnt_up = 0, cnt_dn = 0;
        const int gper = (n_groups + GT - 1) / GT;
        const int gb = min(n_groups, threadIdx.x * gper), ge = min(n_groups, gb + gper);
        for (int g = gb; g < ge; ++g) {
            const bool shared = g >= s_nact;
            const int rows = shared ? a.T : s_cnt[s_act[g]];
            const int mt = (rows + TC_BM - 1) / TC_BM;
            const int fd = shared ? a.Fs : a.F;
            cnt_up += mt * (fd / (TC_BN_UP / 2));
            cnt_dn += mt * n_dn;
        }
        int base_up = block_exclusive_scan(cnt_up, &n_up);
        int base_dn = block_exclusive_scan(cnt_dn, &n_down);
        if (n_up > a.max_up || n_down > a.max_down) {
            if (threadIdx.x == 0) record_error(a.status, DEV_BAD_TILE);
            n_up = n_down = 0;
        } else {
            for (int g = gb; g < ge; ++g) {
                const bool shared = g >= s_nact;
                const int ge_idx = shared ? a.E : s_act[g];
                const int rows = shared ? a.T : s_cnt[ge_idx];
                const int mt = (rows + TC_BM - 1) / TC_BM;
                const int fd = shared ? a.Fs : a.F;
                // (group, n, m) order: tiles sharing a weight tile run side by side
                for (int n = 0; n < fd / (TC_BN_UP / 2); ++n)
                    for (int m = 0; m < mt; ++m)
                        a.up_tiles[base_up++] = TileDesc{ge_idx, m * TC_BM, n * (TC_BN_UP / 2), 0};
                for (int n = 0; n < n_dn; ++n)
                    for (int m = 0; m < mt; ++m)
                        a.down_tiles[base_dn++] = TileDesc{ge_idx, m * TC_BM, n * TC_BN_DOWN, 0};
            }
        }
    }
    if (threadIdx.x == 0) {
        a.meta->n_active = s_nact;
        a.meta->n_up_tiles = n_up;
        a.meta->n_down_tiles = n_down;
        a.meta->n_pairs = a.T * a.K;
        a.meta->ticket = 0;  // ready for the next forward
    }
}

int launch_group(const Layer &L, int T, bool build_tiles, cudaStream_t s)
{
    GroupArgs a;
    a.topk_idx = L.topk_idx;
    a.T = T; a.K = L.K; a.E = L.E; a.Tmax = L.Tmax;
    a.has_shared = L.Fs > 0; a.F = L.F; a.Fs = L.Fs; a.H = L.H;
    a.expert_rows = L.expert_rows; a.counts = L.counts; a.offsets = L.offsets; a.active = L.active;
    a.meta = L.meta;
    a.build_tiles = build_tiles ? 1 : 0;
    a.up_tiles = L.up_tiles; a.down_tiles = L.down_tiles;
    a.max_up = L.max_up_tiles; a.max_down = L.max_down_tiles;
    a.status = L.status;
    group_kernel<<<L.E, GT, 0, s>>>(a);
    return 1;
}

}  // namespace moe
