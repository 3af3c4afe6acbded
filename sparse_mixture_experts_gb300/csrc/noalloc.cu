// noalloc.cu -- moe_route_noalloc: the routing step (router logits, top-k
// selection with routing weights, per-expert token counts) for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a
// caller-managed memory pool or arena that must stay the only owner of device
// memory, in a process whose allocator is locked down after start-up, or in a
// real-time loop where an allocation (and the device-wide synchronisation it
// can imply) is not acceptable.  Such callers cannot create a moe_layer,
// because moe_layer_create allocates the layer's workspace.
//
// The logits between the two kernels live in a file-scope __device__ array of
// NOALLOC_MAX_LOGITS floats (1 MiB) that every GPU which loads the library holds
// until the process exits.  All calls on a device share that array and it keeps
// the last call's contents, so calls that overlap on the GPU (on different
// streams, or from different threads without ordering) race; order them.  The
// per-expert counts are zeroed by the call itself before they are accumulated.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

constexpr size_t NOALLOC_MAX_LOGITS = (size_t)1 << 18;  // 262144 token x expert logits, 1 MiB
constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) float g_noalloc_logits[NOALLOC_MAX_LOGITS];

// Device address of g_noalloc_logits, per device, looked up with that device
// current and kept together with the unique id of the CUDA context it belongs
// to.  A device reset (or a switch to another context) loads the module again
// at another address; the id then differs and the address is looked up anew.
struct NoallocScratch {
    unsigned long long ctx_id = 0;
    float *ptr = nullptr;
};
static NoallocScratch g_noalloc_scratch[NOALLOC_MAX_DEVICES];
static std::mutex g_noalloc_mutex;

typedef int (*PfnCtxGetCurrent)(void **ctx);
typedef int (*PfnCtxGetId)(void *ctx, unsigned long long *id);

// unique id of the calling thread's current CUDA context (0 if unavailable)
static unsigned long long current_context_id()
{
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PfnCtxGetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PfnCtxGetId>(p);
        looked_up = true;
    }
    void *ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
    return id;
}

template <typename TW> __device__ __forceinline__ float load_scalar(const TW *p);
template <> __device__ __forceinline__ float load_scalar<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float load_scalar<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}

// logits[t][e] = Wr[e] . x[t] (+ b[e]); one warp per router row, tokens in
// chunks of 8, blockIdx.y over token ranges
template <typename TW>
__global__ void __launch_bounds__(256) noalloc_logits_kernel(const TW *__restrict__ x, const TW *__restrict__ W,
                                                             const TW *__restrict__ b, int T, int H, int E,
                                                             int tok_per_block, float *__restrict__ logits)
{
    constexpr int V = Vec<TW>::N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    const int tbeg = blockIdx.y * tok_per_block;
    const int tend = min(T, tbeg + tok_per_block);
    const TW *w = W + (size_t)e * H;
    const float bias = b ? load_scalar<TW>(b + e) : 0.0f;
    for (int t0 = tbeg; t0 < tend; t0 += 8) {
        const int nt = min(8, tend - t0);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int c = lane; c < H / V; c += 32) {
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
        for (int j = 0; j < 8; ++j) {
            if (j < nt) {
                const float s = warp_sum(acc[j]);
                if (lane == 0) logits[(size_t)(t0 + j) * E + e] = s + bias;
            }
        }
    }
}

// one warp per token: top-k (ties to the lower index, descending order) and
// routing weights by the same warp routine the layer's selection kernels use,
// and the token's contribution to the per-expert counts
__global__ void __launch_bounds__(256) noalloc_select_kernel(const float *__restrict__ logits, int T, int E, int K,
                                                             int mode, int norm, float scale, int *__restrict__ idx,
                                                             float *__restrict__ wout, int *__restrict__ counts)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    int sel_i;
    float sel_v, w;
    warp_select_any(logits + (size_t)t * E, E, K, mode, norm, scale, lane, sel_i, sel_v, w);
    if (lane < K) {
        idx[(size_t)t * K + lane] = sel_i;
        wout[(size_t)t * K + lane] = w;
        atomicAdd(&counts[sel_i], 1);  // integer: the result does not depend on the order
    }
}

static moe_status na_fail(moe_status st, const char *msg)
{
    set_last_error(msg);
    return st;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_noalloc(const void *x, const void *router_w, const void *router_b, int32_t n_tokens,
                                        int32_t hidden, int32_t n_expert, int32_t top_k, int32_t router_mode,
                                        int32_t norm_topk_prob, float weights_scale, int32_t dtype, int32_t *idx,
                                        float *w, int32_t *counts, void *stream)
{
    set_last_error("");
    if (!x || !router_w || !idx || !w || !counts)
        return na_fail(MOE_ERR_INVALID_ARG, "x, router_w, idx, w and counts must be non-NULL");
    if (n_tokens < 0 || hidden <= 0 || n_expert <= 0 || top_k <= 0)
        return na_fail(MOE_ERR_INVALID_ARG, "sizes must be positive (n_tokens >= 0)");
    if (top_k > n_expert) return na_fail(MOE_ERR_INVALID_ARG, "top_k > n_expert");
    if (top_k > 32 || n_expert > 1024) return na_fail(MOE_ERR_UNSUPPORTED, "top_k > 32 or n_expert > 1024");
    if (hidden % 8) return na_fail(MOE_ERR_UNSUPPORTED, "hidden must be a multiple of 8");
    if (dtype != MOE_DT_F32 && dtype != MOE_DT_BF16) return na_fail(MOE_ERR_INVALID_ARG, "unknown dtype");
    if (router_mode != MOE_ROUTER_SOFTMAX_TOPK && router_mode != MOE_ROUTER_TOPK_SOFTMAX)
        return na_fail(MOE_ERR_INVALID_ARG, "unknown router_mode");
    if (((uintptr_t)x & 15) || ((uintptr_t)router_w & 15))
        return na_fail(MOE_ERR_INVALID_ARG, "x and router_w must be 16-byte aligned");
    if ((size_t)n_tokens * (size_t)n_expert > NOALLOC_MAX_LOGITS)
        return na_fail(MOE_ERR_TOO_MANY_TOKENS,
                       "n_tokens * n_expert exceeds the 262144 logits of the static scratch (1 MiB)");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return na_fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return na_fail(MOE_ERR_UNSUPPORTED, "device ordinal >= 64");
    float *scratch;
    {
        // first call on a device (or in a new context on it): look up the
        // array's device address with that device current; a host-side use of
        // the symbol itself is not a device address
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        NoallocScratch &c = g_noalloc_scratch[dev];
        const unsigned long long id = current_context_id();
        if (!c.ptr || id == 0 || id != c.ctx_id) {
            float *p = nullptr;
            e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_logits);
            if (e != cudaSuccess || !p) return na_fail(MOE_ERR_CUDA, "cudaGetSymbolAddress of the routing scratch failed");
            c.ptr = p;
            // the lookup makes the device's context current if none was
            c.ctx_id = current_context_id();
        }
        scratch = c.ptr;
    }

    cudaStream_t s = (cudaStream_t)stream;
    e = cudaMemsetAsync(counts, 0, (size_t)n_expert * sizeof(int32_t), s);
    if (e != cudaSuccess) return na_fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    if (n_tokens == 0) return MOE_OK;

    int num_sms = 0;
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    const int row_blocks = (n_expert + 7) / 8;
    int tok_per_block = n_tokens;
    if (row_blocks < 2 * num_sms) {
        const int want_y = (2 * num_sms + row_blocks - 1) / row_blocks;
        tok_per_block = ((n_tokens + want_y - 1) / want_y + 7) / 8 * 8;
        if (tok_per_block < 8) tok_per_block = 8;
    }
    const dim3 grid(row_blocks, (n_tokens + tok_per_block - 1) / tok_per_block);
    if (dtype == MOE_DT_BF16)
        noalloc_logits_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)router_w, (const __nv_bfloat16 *)router_b, n_tokens,
            hidden, n_expert, tok_per_block, scratch);
    else
        noalloc_logits_kernel<float><<<grid, 256, 0, s>>>((const float *)x, (const float *)router_w,
                                                          (const float *)router_b, n_tokens, hidden, n_expert,
                                                          tok_per_block, scratch);
    noalloc_select_kernel<<<(n_tokens + 7) / 8, 256, 0, s>>>(scratch, n_tokens, n_expert, top_k, router_mode,
                                                             norm_topk_prob, weights_scale, idx, w, counts);
    e = cudaGetLastError();
    if (e != cudaSuccess) return na_fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    return MOE_OK;
}
