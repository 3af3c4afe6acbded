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
// It is a counting sort in three steps: chunk histograms and in-chunk ranks
// (in the selection kernel), prefixes over chunks and experts (one block), and
// the scatter of each pick to its position.  Everything is integer work with
// a fixed order, so it is deterministic.
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
// selection: one warp per token, SEL_TOK tokens (a "chunk") per block.  Next to
// the picks, each block records, for every expert, how many of the chunk's
// tokens picked it (the chunk histogram, stored expert-major) and, for every
// pick, how many earlier tokens of the chunk picked the same expert (its rank
// within the chunk).  Both come from one SEL_TOK-bit token mask per expert.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(SEL_TOK * 32) select_kernel(float *__restrict__ logits, const float *__restrict__ parts,
                                                              int splits, int T, int E, int R,
                                                              int K, int mode, int norm, float scale, int has_shared,
                                                              int *__restrict__ topk_idx, float *__restrict__ topk_w,
                                                              float *__restrict__ sh_gate, int hist_pitch,
                                                              int *__restrict__ chunk_hist, int *__restrict__ pair_rank)
{
    __shared__ uint32_t s_tm[1024];  // bit w: token w of the chunk picked the expert
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < E; e += SEL_TOK * 32) s_tm[e] = 0u;
    __syncthreads();
    const int t = blockIdx.x * SEL_TOK + warp;
    int sel_i = -1;
    if (t < T && splits > 1) {
        // the router GEMM split K: its partial sums, added in split order, are the logits
        for (int e = lane; e < R; e += 32) {
            float p[TC_ROUTER_MAX_SPLITS];
#pragma unroll
            for (int sp = 0; sp < TC_ROUTER_MAX_SPLITS; ++sp)
                p[sp] = sp < splits ? __ldcg(parts + ((size_t)sp * T + t) * R + e) : 0.0f;
            float v = p[0];
#pragma unroll
            for (int sp = 1; sp < TC_ROUTER_MAX_SPLITS; ++sp)
                if (sp < splits) v += p[sp];
            logits[(size_t)t * R + e] = v;
        }
        __syncwarp();
    }
    if (t < T) {
        const float *l = logits + (size_t)t * R;
        float sel_v, w;
        warp_select_any(l, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
        if (lane < K) {
            topk_idx[(size_t)t * K + lane] = sel_i;
            topk_w[(size_t)t * K + lane] = w;
            atomicOr(&s_tm[sel_i], 1u << warp);
        }
        if (has_shared && lane == 0) sh_gate[t] = 1.0f / (1.0f + __expf(-l[E]));
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += SEL_TOK * 32)
        chunk_hist[(size_t)e * hist_pitch + blockIdx.x] = __popc(s_tm[e]);
    if (t < T && lane < K) pair_rank[(size_t)t * K + lane] = __popc(s_tm[sel_i] & ((1u << warp) - 1u));
}

int launch_select(const Layer &L, int T, int splits, cudaStream_t s)
{
    const moe_config &c = L.cfg;
    select_kernel<<<(T + SEL_TOK - 1) / SEL_TOK, SEL_TOK * 32, 0, s>>>(
        L.logits, L.router_parts, splits, T, L.E, L.R, L.K, c.router_mode, c.norm_topk_prob, c.weights_scale,
        L.Fs > 0, L.topk_idx, L.topk_w, L.sh_gate, L.hist_pitch, L.chunk_hist, L.pair_rank);
    return 1;
}

// ---------------------------------------------------------------------------
// grouping plan: one block per expert turns its chunk histogram into where
// each chunk's picks of the expert start (exclusive prefix over chunks) and
// its count; the last block to finish computes the exclusive prefix of the
// counts over experts (each expert's first row in the expert-sorted buffers),
// the list of experts that received tokens, and for the tensor-core path the
// first tile of every group (the active experts, then the shared expert) in
// the gate/up and down tile orders, with each group's expert, rows and first
// row.  The GEMMs map a tile index to its group by walking those firsts, so
// no tile list is written.
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
    int T, K, E, hist_pitch;
    int has_shared, F, Fs, H;
    int *chunk_hist;  // in: [E][hist_pitch] picks per chunk; out: where each chunk's picks start (relative)
    int *counts, *offsets, *active;
    int *gfirst;      // [5][E + 2]: per group first gate/up tile (+ total), first down tile (+ total), expert, rows, first row
    RouteMeta *meta;
    int build_tiles;
    int tm, tnu, tnd; // tile geometry of the expert GEMMs (tc_geometry)
};

__global__ void __launch_bounds__(GT) group_kernel(GroupArgs a)
{
    const int e = blockIdx.x;
    const int tid = threadIdx.x;
    const int nc = (a.T + SEL_TOK - 1) / SEL_TOK;
    int *row = a.chunk_hist + (size_t)e * a.hist_pitch;  // hist_pitch is a multiple of 4

    // exclusive prefix over chunks, four consecutive chunks per thread (one
    // 16-byte load), GT * 4 chunks per pass
    int carry = 0;
    for (int base = 0; base < nc; base += 4 * GT) {
        const int c = base + 4 * tid;
        int4 v = make_int4(0, 0, 0, 0);
        if (c < nc) {
            v = *reinterpret_cast<const int4 *>(row + c);
            if (c + 1 >= nc) v.y = 0;
            if (c + 2 >= nc) v.z = 0;
            if (c + 3 >= nc) v.w = 0;
        }
        int tot;
        const int pre = carry + block_exclusive_scan(v.x + v.y + v.z + v.w, &tot);
        if (c < nc) *reinterpret_cast<int4 *>(row + c) = make_int4(pre, pre + v.x, pre + v.x + v.y, pre + v.x + v.y + v.z);
        carry += tot;
    }

    __shared__ int s_last;
    if (tid == 0) {
        a.counts[e] = carry;
        // release this block's writes, take a ticket; the last block acquires all
        __threadfence();
        s_last = atomicAdd(&a.meta->ticket, 1) == a.E - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last block: offsets, active experts, group tile firsts ----
    __shared__ int s_cnt[1024];
    __shared__ int s_act[1024];
    const int E = a.E;
    for (int i = tid; i < E; i += GT) s_cnt[i] = __ldcg(&a.counts[i]);
    __syncthreads();
    // each thread owns a contiguous run of up to 4 experts (E <= 1024)
    const int per = (E + GT - 1) / GT;
    const int beg = min(E, tid * per), end = min(E, beg + per);
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
    if (tid == 0) a.offsets[E] = tot;
    const int n_act = tot_act;
    __syncthreads();

    int n_up = 0, n_down = 0;
    if (a.build_tiles) {
        const int n_groups = n_act + (a.has_shared ? 1 : 0);  // <= E + 1
        const int n_dn = (a.H + a.tnd - 1) / a.tnd;
        const int gper = (n_groups + GT - 1) / GT;
        const int gb = min(n_groups, tid * gper), ge = min(n_groups, gb + gper);
        int cu = 0, cd = 0;
        for (int g = gb; g < ge; ++g) {
            const bool shared = g >= n_act;
            const int mt = ((shared ? a.T : s_cnt[s_act[g]]) + a.tm - 1) / a.tm;
            cu += mt * (((shared ? a.Fs : a.F) + a.tnu - 1) / a.tnu);
            cd += mt * n_dn;
        }
        int fu = block_exclusive_scan(cu, &n_up);
        int fd = block_exclusive_scan(cd, &n_down);
        int *gu = a.gfirst, *gd = a.gfirst + (E + 2);
        int *gx = a.gfirst + 2 * (E + 2), *gr = a.gfirst + 3 * (E + 2), *g0 = a.gfirst + 4 * (E + 2);
        for (int g = gb; g < ge; ++g) {
            const bool shared = g >= n_act;
            const int rows = shared ? a.T : s_cnt[s_act[g]];
            const int mt = (rows + a.tm - 1) / a.tm;
            gu[g] = fu;
            gd[g] = fd;
            gx[g] = shared ? E : s_act[g];
            gr[g] = rows;
            g0[g] = shared ? a.T * a.K : __ldcg(&a.offsets[s_act[g]]);
            fu += mt * (((shared ? a.Fs : a.F) + a.tnu - 1) / a.tnu);
            fd += mt * n_dn;
        }
        if (tid == 0) { gu[n_groups] = n_up; gd[n_groups] = n_down; }
    }
    if (tid == 0) {
        a.meta->n_active = n_act;
        a.meta->n_up_tiles = n_up;
        a.meta->n_down_tiles = n_down;
        a.meta->n_pairs = a.T * a.K;
        a.meta->ticket = 0;  // ready for the next forward
    }
}

int launch_group(const Layer &L, int T, bool build_tiles, cudaStream_t s)
{
    GroupArgs a;
    a.T = T; a.K = L.K; a.E = L.E; a.hist_pitch = L.hist_pitch;
    a.has_shared = L.Fs > 0; a.F = L.F; a.Fs = L.Fs; a.H = L.H;
    a.chunk_hist = L.chunk_hist;
    a.counts = L.counts; a.offsets = L.offsets; a.active = L.active;
    a.gfirst = L.gfirst;
    a.meta = L.meta;
    a.build_tiles = build_tiles ? 1 : 0;
    const TcGeometry geo = tc_geometry(L, T);
    a.tm = geo.tm; a.tnu = geo.tnu; a.tnd = geo.tnd;
    group_kernel<<<L.E, GT, 0, s>>>(a);
    return 1;
}

// ---------------------------------------------------------------------------
// scatter: the expert-sorted position of pick p = t*K + q of expert e is
// offsets[e] + (start of t's chunk among e's picks) + (its rank in the chunk):
// ascending token order within each expert.  expert_rows[position] = p; with
// rows, also the gather of the token rows into the expert-sorted activation
// buffer (one warp per row).  The shared expert's rows are all tokens in
// order: the gate/up GEMM reads them from x itself.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) scatter_kernel(const __nv_bfloat16 *__restrict__ x, int T, int K, int H,
                                                      int has_shared, int hist_pitch, const int *__restrict__ topk_idx,
                                                      const int *__restrict__ pair_rank,
                                                      const int *__restrict__ chunk_start,
                                                      const int *__restrict__ offsets, int *__restrict__ expert_rows,
                                                      __nv_bfloat16 *__restrict__ xp)
{
    const int P = T * K;
    if (xp == nullptr) {
        // positions only: one thread per pick
        const int p = blockIdx.x * 256 + threadIdx.x;
        if (p >= P) return;
        const int e = topk_idx[p], t = p / K;
        expert_rows[offsets[e] + chunk_start[(size_t)e * hist_pitch + t / SEL_TOK] + pair_rank[p]] = p;
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + warp;
    if (r >= P) return;
    const int e = topk_idx[r];
    const int tok = r / K;
    const int dst = offsets[e] + chunk_start[(size_t)e * hist_pitch + tok / SEL_TOK] + pair_rank[r];
    if (lane == 0) expert_rows[dst] = r;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)tok * H);
    uint4 *d = reinterpret_cast<uint4 *>(xp + (size_t)dst * H);
    // four 16-byte loads in flight per lane before their stores
    const int n16 = H / 8;
    int c = lane;
    for (; c + 96 < n16; c += 128) {
        const uint4 v0 = __ldg(src + c), v1 = __ldg(src + c + 32), v2 = __ldg(src + c + 64), v3 = __ldg(src + c + 96);
        d[c] = v0;
        d[c + 32] = v1;
        d[c + 64] = v2;
        d[c + 96] = v3;
    }
    for (; c < n16; c += 32) d[c] = __ldg(src + c);
}

int launch_scatter(const Layer &L, const void *x, int T, bool rows, cudaStream_t s)
{
    const int P = T * L.K;
    if (!rows) {
        scatter_kernel<<<(P + 255) / 256, 256, 0, s>>>(nullptr, T, L.K, L.H, L.Fs > 0, L.hist_pitch, L.topk_idx,
                                                       L.pair_rank, L.chunk_hist, L.offsets, L.expert_rows, nullptr);
        return 1;
    }
    scatter_kernel<<<(P + 7) / 8, 256, 0, s>>>((const __nv_bfloat16 *)x, T, L.K, L.H, L.Fs > 0, L.hist_pitch,
                                                    L.topk_idx, L.pair_rank, L.chunk_hist, L.offsets, L.expert_rows,
                                                    (__nv_bfloat16 *)L.xp);
    return 1;
}

}  // namespace moe
