// moe_api.cu -- the C ABI of libmoe (declared in include/moe.h).
//
// create : validate the config, copy / repack the weights into library-owned
//          device memory ([out][in] layouts; the gpt-oss interleaved gate_up
//          tensor is split into gate and up tensors, even rows -> gate, odd
//          rows -> up, as "Phase 19: MoE -- gpt-oss-20b", section 2 Experts,
//          defines them; biases are widened to fp32), allocate the workspace.
// forward: router -> select -> group -> experts (weight-streaming or tensor
//          cores) -> combine, all on the caller's stream, nothing allocated.
#include <cstdio>
#include <cstring>
#include <string>

#include "moe_internal.cuh"

using namespace moe;

struct moe_layer : public Layer {};

namespace {

thread_local std::string g_error;

moe_status fail(moe_status st, const std::string &msg)
{
    g_error = msg;
    return st;
}

moe_status cuda_fail(cudaError_t e, const char *what)
{
    g_error = std::string(what) + ": " + cudaGetErrorString(e);
    return e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA;
}

#define CUDA_TRY(call)                                     \
    do {                                                   \
        cudaError_t e_ = (call);                           \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

moe_status dev_alloc(Layer &L, void **p, size_t bytes)
{
    *p = nullptr;
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
        *p = nullptr;
        return cuda_fail(e, "cudaMalloc");
    }
    L.allocations.push_back(*p);
    L.device_bytes += bytes;
    return MOE_OK;
}

template <typename T>
moe_status dev_alloc_t(Layer &L, T **p, size_t count)
{
    return dev_alloc(L, reinterpret_cast<void **>(p), count * sizeof(T));
}

void timing_free(Layer &L)
{
    for (cudaEvent_t e : L.timing_events) cudaEventDestroy(e);
    L.timing_events.clear();
    L.timing_kind.clear();
    L.timing_max = L.timing_recorded = L.timing_pairs = 0;
}

void free_all(Layer &L)
{
    timing_free(L);
    if (L.h2d_stream) {
        cudaStreamSynchronize(L.h2d_stream);
        cudaStreamDestroy(L.h2d_stream);
        L.h2d_stream = nullptr;
    }
    if (L.x_ready) cudaEventDestroy(L.x_ready), L.x_ready = nullptr;
    if (L.x_free) cudaEventDestroy(L.x_free), L.x_free = nullptr;
    residency_release(L);
    if (L.tmaps) tc_release(L);
    if (L.dectc) dectc_release(L);
    for (void *p : L.allocations) cudaFree(p);
    L.allocations.clear();
}

// ---- repacking kernels ------------------------------------------------------
__global__ void widen_kernel(const void *src, int dtype, size_t n, float *dst)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        if (dtype == MOE_DT_BF16) dst[i] = __bfloat162float(((const __nv_bfloat16 *)src)[i]);
        else dst[i] = ((const float *)src)[i];
    }
}

// src [E][2F][H] interleaved (gate = even rows) -> gate [E][F][H], up [E][F][H]
__global__ void deinterleave_rows_kernel(const uint4 *src, size_t rows_2f, size_t row_vecs, uint4 *gate, uint4 *up)
{
    const size_t n = rows_2f * row_vecs;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / row_vecs, c = i - r * row_vecs;
        const size_t dst = (r >> 1) * row_vecs + c;
        if (r & 1) up[dst] = src[i];
        else gate[dst] = src[i];
    }
}

// bias [E][2F] (interleaved or [gate F | up F]) -> fp32 gate_b [E][F], up_b [E][F]
__global__ void split_bias_kernel(const void *src, int dtype, int E, int F, int interleaved, float *gb, float *ub)
{
    const size_t n = (size_t)E * 2 * F;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = dtype == MOE_DT_BF16 ? __bfloat162float(((const __nv_bfloat16 *)src)[i]) : ((const float *)src)[i];
        const size_t e = i / (2 * F), r = i - e * 2 * F;
        size_t f;
        bool is_up;
        if (interleaved) { f = r >> 1; is_up = r & 1; }
        else { f = r % F; is_up = r >= (size_t)F; }
        (is_up ? ub : gb)[e * F + f] = v;
    }
}

// an MXFP4 tensor copied to the device for packing (freed by the caller, cudaFree)
struct Fp4Staged {
    uint8_t *blocks = nullptr, *scales = nullptr;
    void release() { if (blocks) cudaFree(blocks); if (scales) cudaFree(scales); blocks = scales = nullptr; }
};

moe_status stage_mxfp4(const void *blocks, const void *scales, size_t rows, size_t cols, const char *name,
                       Fp4Staged &st)
{
    if (!blocks || !scales) return fail(MOE_ERR_INVALID_ARG, std::string("missing MXFP4 weight: ") + name);
    const size_t nb = cols / 32;
    cudaError_t e = cudaMalloc((void **)&st.blocks, rows * nb * 16);
    if (e == cudaSuccess) e = cudaMalloc((void **)&st.scales, rows * nb);
    if (e == cudaSuccess) e = cudaMemcpy(st.blocks, blocks, rows * nb * 16, cudaMemcpyDefault);
    if (e == cudaSuccess) e = cudaMemcpy(st.scales, scales, rows * nb, cudaMemcpyDefault);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return MOE_OK;
}

// a tensor of Q4 records copied to the device for packing (freed by the caller)
moe_status stage_bytes(const void *src, size_t bytes, const char *name, uint8_t *&dst)
{
    if (!src) return fail(MOE_ERR_INVALID_ARG, std::string("missing Q4 weight: ") + name);
    cudaError_t e = cudaMalloc((void **)&dst, bytes);
    if (e == cudaSuccess) e = cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return MOE_OK;
}

moe_status upload(void *dst, const void *src, size_t bytes, const char *name)
{
    if (!src) return fail(MOE_ERR_INVALID_ARG, std::string("missing weight: ") + name);
    cudaError_t e = cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return MOE_OK;
}

moe_status upload_f32(Layer &L, float **dst, const void *src, size_t n, const char *name)
{
    if (!src) return fail(MOE_ERR_INVALID_ARG, std::string("missing bias: ") + name);
    moe_status st = dev_alloc_t(L, dst, n);
    if (st) return st;
    void *tmp = nullptr;
    CUDA_TRY(cudaMalloc(&tmp, n * L.wbytes));
    cudaError_t e = cudaMemcpy(tmp, src, n * L.wbytes, cudaMemcpyDefault);
    if (e == cudaSuccess) {
        widen_kernel<<<256, 256>>>(tmp, L.cfg.w_dtype, n, *dst);
        e = cudaDeviceSynchronize();
    }
    cudaFree(tmp);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return MOE_OK;
}

moe_status validate(const moe_config &c)
{
    if (c.hidden <= 0 || c.n_expert <= 0 || c.top_k <= 0 || c.expert_ff <= 0 || c.shared_ff < 0 || c.max_tokens < 0)
        return fail(MOE_ERR_INVALID_ARG, "sizes must be positive (shared_ff, max_tokens >= 0)");
    if (c.top_k > c.n_expert) return fail(MOE_ERR_INVALID_ARG, "top_k > n_expert");
    if (c.top_k > 32) return fail(MOE_ERR_UNSUPPORTED, "top_k > 32");
    if (c.n_expert > 1024) return fail(MOE_ERR_UNSUPPORTED, "n_expert > 1024");
    if (c.router_mode != MOE_ROUTER_SOFTMAX_TOPK && c.router_mode != MOE_ROUTER_TOPK_SOFTMAX)
        return fail(MOE_ERR_INVALID_ARG, "unknown router_mode");
    if (c.act != MOE_ACT_SWIGLU && c.act != MOE_ACT_CLAMP_GLU) return fail(MOE_ERR_INVALID_ARG, "unknown act");
    for (int d : {c.act_dtype, c.out_dtype})
        if (d != MOE_DT_F32 && d != MOE_DT_BF16) return fail(MOE_ERR_INVALID_ARG, "unknown dtype");
    if (c.w_dtype != MOE_DT_F32 && c.w_dtype != MOE_DT_BF16 && c.w_dtype != MOE_DT_MXFP4 && c.w_dtype != MOE_DT_Q4)
        return fail(MOE_ERR_INVALID_ARG, "unknown dtype");
    if (c.w_dtype == MOE_DT_MXFP4 || c.w_dtype == MOE_DT_Q4) {
        const std::string f = c.w_dtype == MOE_DT_MXFP4 ? "MXFP4" : "Q4";
        if (c.act_dtype != MOE_DT_BF16) return fail(MOE_ERR_UNSUPPORTED, f + " experts need bf16 activations");
        if (c.w_dtype == MOE_DT_MXFP4 && !c.gate_up_interleaved)
            return fail(MOE_ERR_UNSUPPORTED, "MXFP4 experts need an interleaved gate_up");
        if (c.shared_ff) return fail(MOE_ERR_UNSUPPORTED, f + " experts need a layer without a shared expert");
        if (c.hidden % 64 || c.expert_ff % 64)
            return fail(MOE_ERR_UNSUPPORTED, f + " experts need hidden and expert_ff multiples of 64");
    } else if (c.act_dtype != c.w_dtype) {
        return fail(MOE_ERR_UNSUPPORTED, "act_dtype must equal w_dtype");
    }
    if (c.hidden % 8 || c.expert_ff % 8 || c.shared_ff % 8)
        return fail(MOE_ERR_UNSUPPORTED, "hidden, expert_ff and shared_ff must be multiples of 8");
    if ((long long)c.max_tokens * c.top_k > (1LL << 30)) return fail(MOE_ERR_UNSUPPORTED, "max_tokens too large");
    if (c.resident_experts < 0 || (c.resident_experts > 0 && c.resident_experts >= c.n_expert))
        return fail(MOE_ERR_INVALID_ARG, "resident_experts must be 0 or below n_expert");
    if (c.resident_experts > 0) {
        // a chunk of 16 tokens must find a slot for every expert it selects
        const int most = c.n_expert < 16 * c.top_k ? c.n_expert : 16 * c.top_k;
        if (c.resident_experts < most)
            return fail(MOE_ERR_INVALID_ARG, "resident_experts below min(n_expert, 16 * top_k)");
        if (c.w_dtype == MOE_DT_F32) return fail(MOE_ERR_UNSUPPORTED, "expert residency needs bf16 or low-bit experts");
    }
    return MOE_OK;
}

moe_status create_impl(const moe_config *cfg, const moe_weights *w, Layer &L)
{
    moe_status st = validate(*cfg);
    if (st) return st;
    // a low-bit layer keeps its routed experts packed only; every other tensor
    // of it is bf16
    L.qfmt = cfg->w_dtype == MOE_DT_MXFP4 ? QF_MXFP4 : cfg->w_dtype == MOE_DT_Q4 ? QF_Q4 : QF_NONE;
    moe_config cb = *cfg;
    if (L.qfmt != QF_NONE) cb.w_dtype = MOE_DT_BF16;
    const moe_config &c = cb;
    L.cfg = c;
    CUDA_TRY(cudaGetDevice(&L.device));
    CUDA_TRY(cudaDeviceGetAttribute(&L.num_sms, cudaDevAttrMultiProcessorCount, L.device));
    L.E = c.n_expert; L.H = c.hidden; L.F = c.expert_ff; L.Fs = c.shared_ff; L.K = c.top_k;
    L.R = L.E + (L.Fs > 0 ? 1 : 0);
    L.Fmax = L.F > L.Fs ? L.F : L.Fs;
    L.Tmax = c.max_tokens > 0 ? c.max_tokens : 1;
    L.S = c.resident_experts;
    L.wslots = L.E;
    L.wbytes = c.w_dtype == MOE_DT_BF16 ? 2 : 4;
    const size_t E = L.E, H = L.H, F = L.F, Fs = L.Fs, K = L.K, T = L.Tmax, eb = L.wbytes;

    if (!w->router_w || !w->down_w) return fail(MOE_ERR_INVALID_ARG, "missing router_w or down_w");
    if (c.gate_up_interleaved ? !w->gate_up_w : (!w->gate_w || !w->up_w))
        return fail(MOE_ERR_INVALID_ARG, "missing gate/up weights");
    if (c.has_bias && (!w->router_b || !w->gate_up_b || !w->down_b))
        return fail(MOE_ERR_INVALID_ARG, "has_bias set but a bias is missing");
    if (Fs && (!w->sh_gate_w || !w->sh_up_w || !w->sh_down_w || !w->sh_gate_inp))
        return fail(MOE_ERR_INVALID_ARG, "shared_ff > 0 but a shared-expert weight is missing");

    // ---- weights ----
    if ((st = dev_alloc(L, &L.router_w, (size_t)L.R * H * eb))) return st;
    if ((st = upload(L.router_w, w->router_w, E * H * eb, "router_w"))) return st;
    if (Fs && (st = upload((char *)L.router_w + E * H * eb, w->sh_gate_inp, H * eb, "sh_gate_inp"))) return st;
    Fp4Staged gu4, dn4;  // the MXFP4 tensors on the device until the packing below
    Fp4Staged q4a, q4b;  // Q4 records: (gate_up or gate, up), (down, -)
    struct Release {
        Fp4Staged &a, &b, &c, &d;
        ~Release() { a.release(); b.release(); c.release(); d.release(); }
    } release_fp4{gu4, dn4, q4a, q4b};
    if (L.qfmt == QF_MXFP4) {
        // the routed experts stay MXFP4: the tensor-core kernels widen them on chip
        if ((st = stage_mxfp4(w->gate_up_w, w->gate_up_scales, E * 2 * F, H, "gate_up_w", gu4))) return st;
        if ((st = stage_mxfp4(w->down_w, w->down_scales, E * H, F, "down_w", dn4))) return st;
    } else if (L.qfmt == QF_Q4) {
        // the routed experts stay Q4 records, 18 bytes per 32 elements of a row
        if (c.gate_up_interleaved) {
            if ((st = stage_bytes(w->gate_up_w, E * 2 * F * (H / 32) * 18, "gate_up_w", q4a.blocks))) return st;
        } else {
            if ((st = stage_bytes(w->gate_w, E * F * (H / 32) * 18, "gate_w", q4a.blocks))) return st;
            if ((st = stage_bytes(w->up_w, E * F * (H / 32) * 18, "up_w", q4a.scales))) return st;
        }
        if ((st = stage_bytes(w->down_w, E * H * (F / 32) * 18, "down_w", q4b.blocks))) return st;
    } else {
        if ((st = dev_alloc(L, &L.gate_w, E * F * H * eb))) return st;
        if ((st = dev_alloc(L, &L.up_w, E * F * H * eb))) return st;
    }
    if (L.qfmt != QF_NONE) {
        // nothing more: the packed blocks are built below
    } else if (c.gate_up_interleaved) {
        void *tmp = nullptr;
        CUDA_TRY(cudaMalloc(&tmp, E * 2 * F * H * eb));
        cudaError_t e = cudaMemcpy(tmp, w->gate_up_w, E * 2 * F * H * eb, cudaMemcpyDefault);
        if (e == cudaSuccess) {
            deinterleave_rows_kernel<<<4 * L.num_sms, 256>>>((const uint4 *)tmp, E * 2 * F, H * eb / 16,
                                                             (uint4 *)L.gate_w, (uint4 *)L.up_w);
            e = cudaDeviceSynchronize();
        }
        cudaFree(tmp);
        if (e != cudaSuccess) return cuda_fail(e, "gate_up_w");
    } else {
        if ((st = upload(L.gate_w, w->gate_w, E * F * H * eb, "gate_w"))) return st;
        if ((st = upload(L.up_w, w->up_w, E * F * H * eb, "up_w"))) return st;
    }
    if (L.qfmt == QF_NONE) {
        if ((st = dev_alloc(L, &L.down_w, E * H * F * eb))) return st;
        if ((st = upload(L.down_w, w->down_w, E * H * F * eb, "down_w"))) return st;
    }
    if (c.has_bias) {
        if ((st = upload_f32(L, &L.router_b, w->router_b, E, "router_b"))) return st;
        if ((st = upload_f32(L, &L.down_b, w->down_b, E * H, "down_b"))) return st;
        if ((st = dev_alloc_t(L, &L.gate_b, E * F))) return st;
        if ((st = dev_alloc_t(L, &L.up_b, E * F))) return st;
        void *tmp = nullptr;
        CUDA_TRY(cudaMalloc(&tmp, E * 2 * F * eb));
        cudaError_t e = cudaMemcpy(tmp, w->gate_up_b, E * 2 * F * eb, cudaMemcpyDefault);
        if (e == cudaSuccess) {
            split_bias_kernel<<<256, 256>>>(tmp, c.w_dtype, L.E, L.F, c.gate_up_interleaved, L.gate_b, L.up_b);
            e = cudaDeviceSynchronize();
        }
        cudaFree(tmp);
        if (e != cudaSuccess) return cuda_fail(e, "gate_up_b");
    }
    if (Fs) {
        if ((st = dev_alloc(L, &L.sh_gate_w, Fs * H * eb))) return st;
        if ((st = dev_alloc(L, &L.sh_up_w, Fs * H * eb))) return st;
        if ((st = dev_alloc(L, &L.sh_down_w, H * Fs * eb))) return st;
        if ((st = upload(L.sh_gate_w, w->sh_gate_w, Fs * H * eb, "sh_gate_w"))) return st;
        if ((st = upload(L.sh_up_w, w->sh_up_w, Fs * H * eb, "sh_up_w"))) return st;
        if ((st = upload(L.sh_down_w, w->sh_down_w, H * Fs * eb, "sh_down_w"))) return st;
    }

    // ---- workspace ----
    if ((st = dev_alloc_t(L, &L.logits, T * L.R))) return st;
    if ((st = dev_alloc_t(L, &L.topk_idx, T * K))) return st;
    if ((st = dev_alloc_t(L, &L.topk_w, T * K))) return st;
    if ((st = dev_alloc_t(L, &L.sh_gate, T))) return st;
    if ((st = dev_alloc_t(L, &L.counts, E))) return st;
    if ((st = dev_alloc_t(L, &L.offsets, E + 1))) return st;
    if ((st = dev_alloc_t(L, &L.expert_rows, T * K))) return st;
    L.hist_pitch = (int)(((T + SEL_TOK - 1) / SEL_TOK + 3) / 4 * 4);
    if ((st = dev_alloc_t(L, &L.chunk_hist, E * (size_t)L.hist_pitch))) return st;
    if ((st = dev_alloc_t(L, &L.pair_rank, T * K))) return st;
    if ((st = dev_alloc_t(L, &L.active, E))) return st;
    if ((st = dev_alloc_t(L, &L.meta, 1))) return st;
    if ((st = dev_alloc(L, &L.h, (T * K + T) * (size_t)L.Fmax * eb))) return st;
    if ((st = dev_alloc_t(L, &L.ys, T * (K + 1) * H))) return st;
    if ((st = dev_alloc_t(L, &L.status, 1))) return st;
    if ((st = dev_alloc_t(L, &L.never, 1))) return st;
    CUDA_TRY(cudaMemset(L.never, 0, sizeof(int)));
    if ((st = dev_alloc_t(L, &L.gbar, 2))) return st;
    if ((st = dev_alloc(L, &L.x_stage, T * H * eb))) return st;
    if ((st = dev_alloc(L, &L.out_stage, T * H * (c.out_dtype == MOE_DT_BF16 ? 2 : 4)))) return st;
    CUDA_TRY(cudaMemset(L.meta, 0, sizeof(RouteMeta)));
    CUDA_TRY(cudaMemset(L.status, 0, sizeof(int)));
    CUDA_TRY(cudaMemset(L.gbar, 0, 2 * sizeof(unsigned)));
    decode_prepare(L);
    CUDA_TRY(cudaMemset(L.counts, 0, E * sizeof(int)));

    std::string why;
    L.tc_capable = tc_supported(L, why);
    if (L.qfmt != QF_NONE) {
        L.decode_grid = 0;  // the CUDA-core paths read bf16 or fp32 weights only
        if (!L.tc_capable) return fail(MOE_ERR_UNSUPPORTED, "low-bit experts need the tensor-core kernels: " + why);
    }
    if (L.tc_capable) {
        // routed rows (T*K, expert-sorted) then the shared expert's rows (T)
        if ((st = dev_alloc(L, &L.xp, (T * K + T) * H * eb))) return st;
        if ((st = dev_alloc_t(L, &L.gfirst, 5 * (E + 2)))) return st;
        if ((st = dev_alloc_t(L, &L.router_parts, (size_t)TC_ROUTER_MAX_SPLITS * T * L.R))) return st;
        // bf16 experts move to host memory before any tensor map names them
        if (L.S > 0 && L.qfmt == QF_NONE && (st = residency_setup(L))) return st;
        if (tc_prepare(L) != 0) return fail(MOE_ERR_CUDA, "tensor map creation failed");
        if (L.qfmt != QF_NONE) {
            // one contiguous block per (row block, 64-wide K block) for both
            // tensor-core paths
            if ((st = dev_alloc_t(L, &L.fp4_gu, dectc_fp4_bytes(L, true)))) return st;
            if ((st = dev_alloc_t(L, &L.fp4_dn, dectc_fp4_bytes(L, false)))) return st;
            if (L.qfmt == QF_MXFP4 && dectc_pack_fp4(L, gu4.blocks, gu4.scales, dn4.blocks, dn4.scales) != 0)
                return fail(MOE_ERR_CUDA, "MXFP4 packing failed");
            if (L.qfmt == QF_Q4 &&
                dectc_pack_q4(L, c.gate_up_interleaved ? q4a.blocks : nullptr,
                              c.gate_up_interleaved ? nullptr : q4a.blocks, q4a.scales, q4b.blocks) != 0)
                return fail(MOE_ERR_CUDA, "Q4 packing failed");
            if (L.S > 0 && (st = residency_setup(L))) return st;
        }
        size_t hp_b, part_b, tab_b, tick_b;
        dectc_workspace(L, hp_b, part_b, tab_b, tick_b);
        if ((st = dev_alloc(L, &L.dec_hp, hp_b))) return st;
        if ((st = dev_alloc(L, (void **)&L.dec_partials, part_b))) return st;
        if ((st = dev_alloc(L, (void **)&L.dec_wtab, tab_b))) return st;
        if ((st = dev_alloc(L, (void **)&L.dec_tickets, tick_b))) return st;
        CUDA_TRY(cudaMemset(L.dec_tickets, 0, tick_b));
        CUDA_TRY(cudaMemset(L.dec_hp, 0, hp_b));
        if (dectc_prepare(L) != 0) return fail(MOE_ERR_CUDA, "decode tensor map creation failed");
    }
    if (L.S > 0 && !L.dectc)
        return fail(MOE_ERR_UNSUPPORTED, "expert residency needs the weight-streaming tensor-core kernels: " + why);
    CUDA_TRY(cudaDeviceSynchronize());
    return MOE_OK;
}

enum class Route { DecodeTC, Fused, TC, Stream };

Route choose_path(const Layer &L, int T)
{
    switch (L.path) {
    case MOE_PATH_DECODE_TC: return Route::DecodeTC;
    case MOE_PATH_FUSED: return Route::Fused;
    case MOE_PATH_TC: return Route::TC;
    case MOE_PATH_STREAM: return Route::Stream;
    default: break;
    }
    if (dectc_supported(L, T)) return Route::DecodeTC;
    if (decode_supported(L, T)) return Route::Fused;
    if (L.tc_capable) return Route::TC;
    return Route::Stream;
}

// Expert residency: chunks of up to 16 tokens, each through the router, the
// slot assignment and copies of its missing experts, and the weight-streaming
// tensor-core kernel reading the experts through the slot table.
moe_status forward_resident(Layer &L, const void *x, int T, void *out, cudaStream_t s)
{
    const bool rec = L.timing_max > 0 && L.timing_recorded < L.timing_max;
    const size_t xrow = (size_t)L.H * L.wbytes, orow = (size_t)L.H * (L.cfg.out_dtype == MOE_DT_BF16 ? 2 : 4);
    const int kinds[3] = {MOE_KERNEL_ROUTER, MOE_KERNEL_RESIDENCY,
                          L.qfmt == QF_MXFP4 ? MOE_KERNEL_EXPERTS_MXFP4
                                             : L.qfmt == QF_Q4 ? MOE_KERNEL_EXPERTS_Q4 : MOE_KERNEL_EXPERTS};
    int n = 0;
    bool bad = false;
    for (int t0 = 0; t0 < T && !bad; t0 += RESIDENT_CHUNK) {
        const int Tc = T - t0 < RESIDENT_CHUNK ? T - t0 : RESIDENT_CHUNK;
        const void *xc = (const char *)x + (size_t)t0 * xrow;
        void *oc = (char *)out + (size_t)t0 * orow;
        for (int step = 0; step < 3 && !bad; ++step) {
            // per-kernel events while the window has room (a long forward records its first chunks)
            const bool ev = rec && L.timing_pairs < (int)L.timing_kind.size();
            if (ev) {
                cudaEventRecord(L.timing_events[2 * L.timing_pairs], s);
                L.timing_kind[L.timing_pairs] = kinds[step];
            }
            const int r = step == 0   ? launch_dectc(L, xc, Tc, oc, 0, s, t0)
                          : step == 1 ? launch_residency(L, L.logits + (size_t)t0 * L.R, Tc, s)
                                      : launch_dectc(L, xc, Tc, oc, 1, s, t0);
            if (ev) cudaEventRecord(L.timing_events[2 * L.timing_pairs + 1], s), ++L.timing_pairs;
            if (r < 0) bad = true;
            else n += r;
        }
    }
    if (rec) ++L.timing_recorded;
    cudaError_t e = cudaGetLastError();
    if (bad || e != cudaSuccess) return cuda_fail(e != cudaSuccess ? e : cudaErrorLaunchFailure, "resident decode launch");
    L.last_T = T;
    L.last_launches = n;
    L.last_grouped = 0;
    return MOE_OK;
}

moe_status forward_impl(Layer &L, const void *x, int T, void *out, cudaStream_t s)
{
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens < 0");
    if (T > L.cfg.max_tokens) return fail(MOE_ERR_TOO_MANY_TOKENS, "n_tokens > max_tokens");
    if (T == 0) {
        L.last_T = 0;
        L.last_launches = 0;
        return MOE_OK;
    }
    if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x and out must be non-NULL");
    if (((uintptr_t)x & 15) || ((uintptr_t)out & 15)) return fail(MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    const size_t xb = (size_t)T * L.H * L.wbytes;
    const size_t ob = (size_t)T * L.H * (L.cfg.out_dtype == MOE_DT_BF16 ? 2 : 4);
    const char *xs = (const char *)x, *os = (const char *)out;
    if (xs < os + ob && os < xs + xb) return fail(MOE_ERR_INVALID_ARG, "x and out overlap");
    if (L.S > 0) return forward_resident(L, x, T, out, s);
    const Route route = choose_path(L, T);
    if (route == Route::Fused && !decode_supported(L, T))
        return fail(MOE_ERR_UNSUPPORTED, "fused decode path forced for a batch it does not cover");
    if (route == Route::DecodeTC && !dectc_supported(L, T))
        return fail(MOE_ERR_UNSUPPORTED, "weight-streaming tensor-core path forced for a batch it does not cover");
    const bool tc = route == Route::TC;
    const bool rec = L.timing_max > 0 && L.timing_recorded < L.timing_max;
    int n = 0;
    auto run = [&](int kind, auto &&launch) {
        if (rec) {
            cudaEventRecord(L.timing_events[2 * L.timing_pairs], s);
            L.timing_kind[L.timing_pairs] = kind;
        }
        n += launch();
        if (rec) cudaEventRecord(L.timing_events[2 * L.timing_pairs + 1], s), ++L.timing_pairs;
    };
    if (route == Route::DecodeTC) {
        int bad = 0;
        run(MOE_KERNEL_ROUTER, [&] { int r = launch_dectc(L, x, T, out, 0, s); bad |= r < 0; return r < 0 ? 0 : r; });
        run(L.qfmt == QF_MXFP4 ? MOE_KERNEL_EXPERTS_MXFP4 : L.qfmt == QF_Q4 ? MOE_KERNEL_EXPERTS_Q4 : MOE_KERNEL_EXPERTS, [&] { int r = launch_dectc(L, x, T, out, 1, s); bad |= r < 0; return r < 0 ? 0 : r; });
        if (rec) ++L.timing_recorded;
        cudaError_t e = cudaGetLastError();
        if (bad || e != cudaSuccess) return cuda_fail(e != cudaSuccess ? e : cudaErrorLaunchFailure, "decode launch");
        L.last_T = T;
        L.last_launches = n;
        L.last_grouped = 0;
        return MOE_OK;
    }
    if (route == Route::Fused) {
        int launched = 0;
        run(MOE_KERNEL_FUSED, [&] { return launched = launch_decode(L, x, T, out, s); });
        if (launched < 0) {
            cudaError_t e = cudaGetLastError();
            return cuda_fail(e != cudaSuccess ? e : cudaErrorLaunchFailure, "cooperative launch");
        }
        if (rec) ++L.timing_recorded;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        L.last_T = T;
        L.last_launches = n;
        L.last_grouped = 0;
        return MOE_OK;
    }
    int router_bad = 0;
    run(MOE_KERNEL_ROUTER, [&] {
        if (!tc) return launch_router(L, x, T, s);
        const int r = launch_tc_router(L, x, T, s);
        router_bad = r < 0;
        return r < 0 ? 0 : r;
    });
    if (router_bad) return fail(MOE_ERR_CUDA, "tensor map for x could not be encoded");
    const int splits = tc ? tc_router_splits(L, T) : 1;
    run(MOE_KERNEL_SELECT, [&] { return launch_select(L, T, splits, s); });
    run(MOE_KERNEL_GROUP, [&] { return launch_group(L, T, tc, s); });
    run(MOE_KERNEL_GATHER, [&] { return launch_scatter(L, x, T, tc, s); });
    if (tc) {
        int up_bad = 0;
        run(MOE_KERNEL_UP, [&] {
            const int r = launch_experts_tc(L, x, T, 1, s);
            up_bad = r < 0;
            return r < 0 ? 0 : r;
        });
        if (up_bad) return fail(MOE_ERR_CUDA, "tensor map for x could not be encoded");
        run(MOE_KERNEL_DOWN, [&] { return launch_experts_tc(L, x, T, 2, s); });
    } else {
        run(MOE_KERNEL_UP, [&] { return launch_experts_stream(L, x, T, 0, s); });
        run(MOE_KERNEL_DOWN, [&] { return launch_experts_stream(L, x, T, 1, s); });
    }
    run(MOE_KERNEL_COMBINE, [&] { return launch_combine(L, T, out, s); });
    if (rec) ++L.timing_recorded;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    L.last_T = T;
    L.last_launches = n;
    L.last_grouped = 1;
    return MOE_OK;
}

}  // namespace

namespace moe {
// lets other translation units report through moe_last_error()
void set_last_error(const char *msg) { g_error = msg; }
}  // namespace moe

extern "C" {

moe_status moe_layer_create(const moe_config *config, const moe_weights *weights, moe_layer **out)
{
    g_error.clear();
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!config || !weights) return fail(MOE_ERR_INVALID_ARG, "config and weights must be non-NULL");
    moe_layer *L = new (std::nothrow) moe_layer();
    if (!L) return fail(MOE_ERR_OOM, "host allocation failed");
    moe_status st = create_impl(config, weights, *L);
    if (st != MOE_OK) {
        cudaDeviceSynchronize();
        free_all(*L);
        delete L;
        return st;
    }
    *out = L;
    return MOE_OK;
}

moe_status moe_forward(moe_layer *layer, const void *x, int32_t n_tokens, void *out, void *stream)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    return forward_impl(*layer, x, n_tokens, out, (cudaStream_t)stream);
}

moe_status moe_forward_host(moe_layer *layer, const void *x_host, int32_t n_tokens, void *out_host, void *stream)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    Layer &L = *layer;
    if (n_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "n_tokens < 0");
    if (n_tokens > L.cfg.max_tokens) return fail(MOE_ERR_TOO_MANY_TOKENS, "n_tokens > max_tokens");
    if (n_tokens == 0) return forward_impl(L, nullptr, 0, nullptr, (cudaStream_t)stream);
    if (!x_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "x and out must be non-NULL");
    cudaStream_t s = (cudaStream_t)stream;
    const size_t xb = (size_t)n_tokens * L.H * L.wbytes;
    const size_t ob = (size_t)n_tokens * L.H * (L.cfg.out_dtype == MOE_DT_BF16 ? 2 : 4);
    if (!L.h2d_stream) {
        CUDA_TRY(cudaStreamCreateWithFlags(&L.h2d_stream, cudaStreamNonBlocking));
        CUDA_TRY(cudaEventCreateWithFlags(&L.x_ready, cudaEventDisableTiming));
        CUDA_TRY(cudaEventCreateWithFlags(&L.x_free, cudaEventDisableTiming));
        CUDA_TRY(cudaEventRecord(L.x_free, s));  // nothing has read x_stage yet
    }
    // x in on the layer's copy stream, after the last forward that read
    // x_stage, so that the copy overlaps whatever `stream` is still running;
    // `stream` waits for it, so synchronising `stream` covers both copies
    CUDA_TRY(cudaStreamWaitEvent(L.h2d_stream, L.x_free, 0));
    CUDA_TRY(cudaMemcpyAsync(L.x_stage, x_host, xb, cudaMemcpyHostToDevice, L.h2d_stream));
    CUDA_TRY(cudaEventRecord(L.x_ready, L.h2d_stream));
    CUDA_TRY(cudaStreamWaitEvent(s, L.x_ready, 0));
    // A decode batch on the weight-streaming kernel (whose epilogue writes the
    // few KB of out itself) writes straight into out when the host buffer is
    // mapped into the device's address space: no copy out, so nothing sits
    // between this forward and the next one's router on `stream`.  Otherwise
    // out goes through the staging buffer and a copy.
    void *out_dev = nullptr;
    if (L.S > 0 || choose_path(L, n_tokens) == Route::DecodeTC) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, out_host) == cudaSuccess && pa.type == cudaMemoryTypeHost && pa.devicePointer &&
            ((uintptr_t)pa.devicePointer & 15) == 0)
            out_dev = pa.devicePointer;
        else
            cudaGetLastError();  // an unregistered pointer: clear the query's error
    }
    moe_status st = forward_impl(L, L.x_stage, n_tokens, out_dev ? out_dev : L.out_stage, s);
    CUDA_TRY(cudaEventRecord(L.x_free, s));
    if (st) return st;
    if (!out_dev) CUDA_TRY(cudaMemcpyAsync(out_host, L.out_stage, ob, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

moe_status moe_get_routing(moe_layer *layer, int32_t *idx, float *w, void *stream)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    const Layer &L = *layer;
    const size_t n = (size_t)L.last_T * L.K;
    if (n == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (idx) CUDA_TRY(cudaMemcpyAsync(idx, L.topk_idx, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    if (w) CUDA_TRY(cudaMemcpyAsync(w, L.topk_w, n * sizeof(float), cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

moe_status moe_get_logits(moe_layer *layer, float *logits, float *sh_logit, void *stream)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    const Layer &L = *layer;
    if (L.last_T == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (logits)
        CUDA_TRY(cudaMemcpy2DAsync(logits, L.E * sizeof(float), L.logits, L.R * sizeof(float), L.E * sizeof(float),
                                   L.last_T, cudaMemcpyDeviceToDevice, s));
    if (sh_logit && L.Fs > 0)
        CUDA_TRY(cudaMemcpy2DAsync(sh_logit, sizeof(float), L.logits + L.E, L.R * sizeof(float), sizeof(float),
                                   L.last_T, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

moe_status moe_get_expert_counts(moe_layer *layer, int32_t *counts, void *stream)
{
    if (!layer || !counts) return fail(MOE_ERR_INVALID_ARG, "layer and counts must be non-NULL");
    const Layer &L = *layer;
    CUDA_TRY(cudaMemcpyAsync(counts, L.counts, L.E * sizeof(int32_t), cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_get_intermediate(moe_layer *layer, int32_t which, void *dst, size_t capacity, size_t *size,
                                void *stream)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    const Layer &L = *layer;
    const size_t T = (size_t)L.last_T, K = (size_t)L.K;
    const size_t rows = T * K + (L.Fs > 0 ? T : 0);
    const void *src = nullptr;
    size_t bytes = 0;
    switch (which) {
    case MOE_INTER_OFFSETS: src = L.offsets; bytes = T ? ((size_t)L.E + 1) * sizeof(int32_t) : 0; break;
    case MOE_INTER_PERM: src = L.expert_rows; bytes = T * K * sizeof(int32_t); break;
    case MOE_INTER_H: src = L.h; bytes = rows * (size_t)L.Fmax * L.wbytes; break;
    case MOE_INTER_YS: src = L.ys; bytes = T * (K + 1) * (size_t)L.H * sizeof(float); break;
    default: return fail(MOE_ERR_INVALID_ARG, "unknown intermediate");
    }
    if (size) *size = bytes;
    if (bytes == 0 || !dst) return MOE_OK;
    if (!L.last_grouped)
        return fail(MOE_ERR_UNSUPPORTED, "the last forward ran a decode path, which keeps no grouped intermediates");
    if (capacity < bytes) return fail(MOE_ERR_INVALID_ARG, "destination too small");
    CUDA_TRY(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
    return MOE_OK;
}

moe_status moe_set_path(moe_layer *layer, int32_t path)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    if (path < MOE_PATH_AUTO || path > MOE_PATH_DECODE_TC) return fail(MOE_ERR_INVALID_ARG, "unknown path");
    if (path == MOE_PATH_DECODE_TC && !layer->dectc)
        return fail(MOE_ERR_UNSUPPORTED, "weight-streaming tensor-core path unavailable (needs the tensor-core path)");
    if (path == MOE_PATH_FUSED && layer->decode_grid == 0)
        return fail(MOE_ERR_UNSUPPORTED, layer->qfmt != QF_NONE ? "low-bit experts run on the tensor-core paths only"
                                                                : "cooperative launch unavailable on this device");
    if (path == MOE_PATH_STREAM && layer->qfmt != QF_NONE)
        return fail(MOE_ERR_UNSUPPORTED, "low-bit experts run on the tensor-core paths only");
    if (layer->S > 0 && path != MOE_PATH_AUTO && path != MOE_PATH_DECODE_TC)
        return fail(MOE_ERR_UNSUPPORTED, "a layer with streamed experts runs the weight-streaming tensor-core path only");
    if (path == MOE_PATH_TC && !layer->tc_capable) {
        std::string why;
        tc_supported(*layer, why);
        return fail(MOE_ERR_UNSUPPORTED, "tensor-core path unavailable: " + why);
    }
    layer->path = path;
    return MOE_OK;
}

moe_status moe_timing_enable(moe_layer *layer, int32_t max_forwards)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    if (max_forwards < 0 || max_forwards > 4096) return fail(MOE_ERR_INVALID_ARG, "max_forwards out of range");
    Layer &L = *layer;
    CUDA_TRY(cudaDeviceSynchronize());
    timing_free(L);
    if (max_forwards == 0) return MOE_OK;
    const size_t pairs = (size_t)max_forwards * MAX_LAUNCHES_PER_FORWARD;
    L.timing_events.resize(2 * pairs);
    for (size_t i = 0; i < 2 * pairs; ++i) {
        cudaError_t e = cudaEventCreate(&L.timing_events[i]);
        if (e != cudaSuccess) {
            L.timing_events.resize(i);
            timing_free(L);
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    L.timing_kind.assign(pairs, 0);
    L.timing_max = max_forwards;
    return MOE_OK;
}

moe_status moe_timing_read(moe_layer *layer, float *total_ms, int32_t *launches)
{
    if (!layer || !total_ms || !launches) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    Layer &L = *layer;
    if (L.timing_max == 0) return fail(MOE_ERR_INVALID_ARG, "timing is not enabled");
    CUDA_TRY(cudaDeviceSynchronize());
    for (int k = 0; k < MOE_KERNEL_COUNT; ++k) { total_ms[k] = 0.0f; launches[k] = 0; }
    for (int p = 0; p < L.timing_pairs; ++p) {
        float ms = 0.0f;
        CUDA_TRY(cudaEventElapsedTime(&ms, L.timing_events[2 * p], L.timing_events[2 * p + 1]));
        total_ms[L.timing_kind[p]] += ms;
        launches[L.timing_kind[p]] += 1;
    }
    L.timing_pairs = 0;
    L.timing_recorded = 0;
    return MOE_OK;
}

moe_status moe_get_status(moe_layer *layer)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    CUDA_TRY(cudaDeviceSynchronize());
    int code = 0;
    CUDA_TRY(cudaMemcpy(&code, layer->status, sizeof(int), cudaMemcpyDeviceToHost));
    if (code != 0) {
        // a kernel that gave up may have left its inter-block counters mid-count:
        // start the next forward from zero
        Layer &L = *layer;
        CUDA_TRY(cudaMemset(L.gbar, 0, 2 * sizeof(unsigned)));
        CUDA_TRY(cudaMemset(L.meta, 0, sizeof(RouteMeta)));
        if (L.dec_tickets) {
            size_t hp_b, part_b, tab_b, tick_b;
            dectc_workspace(L, hp_b, part_b, tab_b, tick_b);
            CUDA_TRY(cudaMemset(L.dec_tickets, 0, tick_b));
        }
        CUDA_TRY(cudaDeviceSynchronize());
        CUDA_TRY(cudaMemset(layer->status, 0, sizeof(int)));
        char buf[96];
        snprintf(buf, sizeof buf, "device-side error %d recorded by a kernel", code);
        return fail(code == DEV_BAD_TILE ? MOE_ERR_CUDA : MOE_ERR_DEVICE_TIMEOUT, buf);
    }
    return MOE_OK;
}

moe_status moe_set_wait_limit(moe_layer *layer, int64_t ns)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    if (ns > 10000000000LL) return fail(MOE_ERR_INVALID_ARG, "wait limit above 10 s");
    layer->wait_ns = ns <= 0 ? 1000000000ull : (unsigned long long)(ns < 1000 ? 1000 : ns);
    return MOE_OK;
}

moe_status moe_set_fault_injection(moe_layer *layer, int32_t on)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    layer->inject = on ? 1 : 0;
    return MOE_OK;
}

int32_t moe_last_launch_count(const moe_layer *layer) { return layer ? layer->last_launches : 0; }
int32_t moe_last_token_count(const moe_layer *layer) { return layer ? layer->last_T : 0; }

size_t moe_device_bytes(const moe_layer *layer) { return layer ? layer->device_bytes : 0; }

void moe_destroy(moe_layer *layer)
{
    if (!layer) return;
    cudaDeviceSynchronize();
    free_all(*layer);
    delete layer;
}

moe_status moe_get_residency(moe_layer *layer, int32_t *expert_of, int64_t *stats)
{
    if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    set_last_error("");
    return residency_read(*layer, expert_of, stats);
}

const char *moe_last_error(void) { return g_error.c_str(); }

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

}  // extern "C"
