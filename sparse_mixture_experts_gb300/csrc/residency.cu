// residency.cu -- expert residency: a bounded set of device slots for the
// routed experts, the rest streamed in from pinned host memory on demand
// ("Engine" (cherenkov), sections "Decode and expert IO" (a pool of resident
// experts, the others read in when a token needs them, expert addresses
// resolved through a table) and "Memory ownership" (expert pools own their
// slot memory)).
//
// On GB300 the host memory is the Grace CPU's, reached from the GPU over the
// chip-to-chip link: the copies are plain 16-byte loads of mapped pinned
// memory by a kernel, so nothing waits for the host.  Per chunk of up to 16
// tokens:
//   1. residency_kernel (one block) recomputes the chunk's selection from the
//      router logits with the decode kernel's own routine, stamps the slots
//      of the selected experts that are resident (hits), and gives each
//      missing expert, in ascending expert order, the least recently used
//      slot among those no expert of the chunk needs (ties: the lower slot):
//      the slots are sorted once by (stamp, slot) and the misses take the
//      first ones.  It writes the copy list and updates the tables.
//   2. stream_experts_kernel copies each missing expert's weight regions
//      from host memory into its slot.
//   3. the weight-streaming decode kernel reads each selected expert through
//      slot_of.
// Every slot a miss can take has a stamp below the chunk's (the layer needs
// S >= the most experts a chunk can select), so the assignment never fails.
#include "moe_internal.cuh"

namespace moe {

constexpr int RES_THREADS = 1024;
constexpr int RES_MAX_SLOTS = 1024;
constexpr int RES_MAX_TOK = 16;  // tokens per chunk (the decode kernel's N)

struct ResArgs {
    const float *logits;  // [T][R] of the chunk
    int T, E, K, R, S, mode, norm;
    float scale;
    int *slot_of;         // [E]
    int *expert_of;       // [S]
    unsigned *last_used;  // [S]
    int *jobs;            // [1 + 2S]
    unsigned long long *stats;  // [4] hits, misses, bytes, chunks
    unsigned long long bytes_per_expert;
    int *status;
};

__global__ void __launch_bounds__(RES_THREADS, 1) residency_kernel(const ResArgs a)
{
    __shared__ uint32_t s_sel[32];                 // bit e: expert e selected in the chunk (E <= 1024)
    __shared__ uint32_t s_miss[32];                // bit e: selected and not resident
    __shared__ unsigned long long s_key[RES_MAX_SLOTS];
    __shared__ int s_hits;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E, S = a.S;
    const unsigned stamp = (unsigned)a.stats[3] + 1u;  // this chunk (stamps start at 1; slots at 0)
    if (tid < 32) s_sel[tid] = s_miss[tid] = 0u;
    if (tid == 0) s_hits = 0;
    __syncthreads();

    // 1. the chunk's selection: the decode kernel's routine, two tokens per warp
    constexpr int NW = RES_THREADS / 32;
    for (int t = warp; t < a.T; t += 2 * NW) {
        const int t2 = t + NW;
        const bool two = t2 < a.T;
        int sel_i[2];
        float sel_v[2], w[2];
        warp_select2_any(a.logits + (size_t)t * a.R, a.logits + (size_t)(two ? t2 : t) * a.R, E, a.K, a.mode,
                         a.norm, a.scale, lane, sel_i, sel_v, w);
        if (lane < a.K) {
            atomicOr(&s_sel[sel_i[0] >> 5], 1u << (sel_i[0] & 31));
            if (two) atomicOr(&s_sel[sel_i[1] >> 5], 1u << (sel_i[1] & 31));
        }
    }
    __syncthreads();

    // 2. hits: stamp their slots; misses: a bit mask
    int my_hits = 0;
    for (int e = tid; e < E; e += RES_THREADS) {
        if (!((s_sel[e >> 5] >> (e & 31)) & 1u)) continue;
        const int slot = a.slot_of[e];
        if (slot >= 0) {
            a.last_used[slot] = stamp;
            ++my_hits;
        } else {
            atomicOr(&s_miss[e >> 5], 1u << (e & 31));
        }
    }
    if (my_hits) atomicAdd(&s_hits, my_hits);
    __syncthreads();

    // 3. the slots ordered by (stamp, slot): ascending bitonic sort of the
    //    keys, padded to a power of two with the largest key
    int P = 1;
    while (P < S) P <<= 1;
    for (int i = tid; i < P; i += RES_THREADS)
        s_key[i] = i < S ? ((unsigned long long)a.last_used[i] << 32) | (unsigned)i : ~0ull;
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P; i += RES_THREADS) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long x = s_key[i], y = s_key[l];
                    const bool up = (i & k) == 0;
                    if (up ? x > y : x < y) {
                        s_key[i] = y;
                        s_key[l] = x;
                    }
                }
            }
            __syncthreads();
        }
    }

    // 4. the n-th miss (ascending expert) takes the n-th slot of that order
    int nmiss = 0;
    for (int wd = 0; wd < 32; ++wd) nmiss += __popc(s_miss[wd]);
    for (int e = tid; e < E; e += RES_THREADS) {
        const uint32_t m = s_miss[e >> 5];
        if (!((m >> (e & 31)) & 1u)) continue;
        int r = __popc(m & ((1u << (e & 31)) - 1u));
        for (int wd = 0; wd < (e >> 5); ++wd) r += __popc(s_miss[wd]);
        const unsigned long long key = r < S ? s_key[r] : ~0ull;
        const int v = (int)(key & 0xffffffffu);
        if (r >= S || (unsigned)(key >> 32) >= stamp) {
            // no free slot: cannot happen when S covers a chunk's selection
            record_error(a.status, DEV_NOT_RESIDENT);
            continue;
        }
        const int old = a.expert_of[v];
        if (old >= 0) a.slot_of[old] = -1;
        a.expert_of[v] = e;
        a.slot_of[e] = v;
        a.last_used[v] = stamp;
        a.jobs[1 + 2 * r] = e;
        a.jobs[2 + 2 * r] = v;
    }
    if (tid == 0) {
        a.jobs[0] = nmiss;
        a.stats[0] += (unsigned long long)s_hits;
        a.stats[1] += (unsigned long long)nmiss;
        a.stats[2] += (unsigned long long)nmiss * a.bytes_per_expert;
        a.stats[3] = stamp;
    }
}

struct StreamArgs {
    const int *jobs;
    const uint8_t *src[3];  // pinned host copies, region r of expert e at src[r] + e * bytes[r]
    uint8_t *dst[3];        // device slots, region r of slot v at dst[r] + v * bytes[r]
    unsigned long long vec[3];  // 16-byte vectors per expert of each region
    unsigned long long per_job; // their sum
    int n_regions;
};

// The copies of a chunk's misses, each a flat range of 16-byte vectors over
// the expert's regions; four independent host loads in flight per thread.
__global__ void __launch_bounds__(256) stream_experts_kernel(const StreamArgs a)
{
    const unsigned long long n = (unsigned long long)a.jobs[0] * a.per_job;
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    for (unsigned long long i0 = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += 4 * stride) {
        uint4 v[4];
        uint4 *d[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            d[u] = nullptr;
            const unsigned long long i = i0 + u * stride;
            if (i >= n) continue;
            const unsigned long long j = i / a.per_job;
            unsigned long long c = i - j * a.per_job;
            int r = 0;
            while (r + 1 < a.n_regions && c >= a.vec[r]) c -= a.vec[r++];
            const int e = a.jobs[1 + 2 * j], slot = a.jobs[2 + 2 * j];
            v[u] = reinterpret_cast<const uint4 *>(a.src[r])[(unsigned long long)e * a.vec[r] + c];
            d[u] = reinterpret_cast<uint4 *>(a.dst[r]) + (unsigned long long)slot * a.vec[r] + c;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (d[u]) *d[u] = v[u];
    }
}

namespace {
moe_status res_fail(moe_status st, const char *msg)
{
    set_last_error(msg);
    return st;
}
}  // namespace

// At create, once the weight arrays hold every expert in their final (packed)
// form: copy each region to pinned host memory, keep experts 0 .. S-1 in S
// device slots and free the full device arrays.
moe_status residency_setup(Layer &L)
{
    const int E = L.E, S = L.S;
    void **arr[3];
    if (L.qfmt != QF_NONE) {
        L.n_regions = 2;
        arr[0] = (void **)&L.fp4_gu;
        arr[1] = (void **)&L.fp4_dn;
        L.region_bytes[0] = dectc_fp4_bytes(L, true) / E;
        L.region_bytes[1] = dectc_fp4_bytes(L, false) / E;
    } else {
        L.n_regions = 3;
        arr[0] = &L.gate_w;
        arr[1] = &L.up_w;
        arr[2] = &L.down_w;
        L.region_bytes[0] = L.region_bytes[1] = L.region_bytes[2] = (size_t)L.F * L.H * L.wbytes;
    }
    for (int r = 0; r < L.n_regions; ++r) {
        const size_t per = L.region_bytes[r];
        if (per % 16) return res_fail(MOE_ERR_UNSUPPORTED, "expert regions must be multiples of 16 bytes");
        cudaError_t e = cudaHostAlloc(&L.host_w[r], (size_t)E * per, cudaHostAllocMapped | cudaHostAllocPortable);
        if (e != cudaSuccess) {
            L.host_w[r] = nullptr;
            return res_fail(MOE_ERR_OOM, "pinned host memory for the streamed experts");
        }
        void *full = *arr[r];
        if ((e = cudaMemcpy(L.host_w[r], full, (size_t)E * per, cudaMemcpyDeviceToHost)) != cudaSuccess)
            return res_fail(MOE_ERR_CUDA, "copy of the experts to host memory");
        void *slots = nullptr;
        if ((e = cudaMalloc(&slots, (size_t)S * per)) != cudaSuccess)
            return res_fail(MOE_ERR_OOM, "expert slots");
        L.allocations.push_back(slots);
        L.device_bytes += (size_t)S * per;
        if ((e = cudaMemcpy(slots, full, (size_t)S * per, cudaMemcpyDeviceToDevice)) != cudaSuccess)
            return res_fail(MOE_ERR_CUDA, "initial expert slots");
        // the full device array is not needed any more
        for (auto it = L.allocations.begin(); it != L.allocations.end(); ++it)
            if (*it == full) {
                L.allocations.erase(it);
                break;
            }
        L.device_bytes -= (size_t)E * per;
        cudaFree(full);
        *arr[r] = slots;
        L.dev_region[r] = slots;
    }
    L.wslots = S;
    // tables: slot s holds expert s
    std::vector<int> slot_of(E), expert_of(S);
    for (int e = 0; e < E; ++e) slot_of[e] = e < S ? e : -1;
    for (int v = 0; v < S; ++v) expert_of[v] = v;
    void *p = nullptr;
    const size_t tab_bytes = (size_t)E * 4 + (size_t)S * 4 + (size_t)S * 4 + (size_t)(1 + 2 * S) * 4 + 4 * 8 + 16;
    if (cudaMalloc(&p, tab_bytes) != cudaSuccess) return res_fail(MOE_ERR_OOM, "residency tables");
    L.allocations.push_back(p);
    L.device_bytes += tab_bytes;
    cudaMemset(p, 0, tab_bytes);
    L.res_stats = (unsigned long long *)p;  // first: 8-byte aligned
    L.slot_of = (int *)(L.res_stats + 4);
    L.expert_of = L.slot_of + E;
    L.last_used = (unsigned *)(L.expert_of + S);
    L.res_jobs = (int *)(L.last_used + S);
    if (cudaMemcpy(L.slot_of, slot_of.data(), (size_t)E * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(L.expert_of, expert_of.data(), (size_t)S * 4, cudaMemcpyHostToDevice) != cudaSuccess)
        return res_fail(MOE_ERR_CUDA, "residency tables");
    return MOE_OK;
}

void residency_release(Layer &L)
{
    for (int r = 0; r < 3; ++r)
        if (L.host_w[r]) {
            cudaFreeHost(L.host_w[r]);
            L.host_w[r] = nullptr;
        }
}

// slot assignment and the copies for one chunk; returns the launches
int launch_residency(const Layer &L, const float *logits, int T, cudaStream_t s)
{
    ResArgs a;
    a.logits = logits;
    a.T = T; a.E = L.E; a.K = L.K; a.R = L.R; a.S = L.S;
    a.mode = L.cfg.router_mode; a.norm = L.cfg.norm_topk_prob; a.scale = L.cfg.weights_scale;
    a.slot_of = L.slot_of; a.expert_of = L.expert_of; a.last_used = L.last_used; a.jobs = L.res_jobs;
    a.stats = L.res_stats;
    unsigned long long per = 0;
    for (int r = 0; r < L.n_regions; ++r) per += L.region_bytes[r];
    a.bytes_per_expert = per;
    a.status = L.status;
    residency_kernel<<<1, RES_THREADS, 0, s>>>(a);
    StreamArgs b;
    b.jobs = L.res_jobs;
    b.n_regions = L.n_regions;
    b.per_job = 0;
    for (int r = 0; r < 3; ++r) {
        b.src[r] = (const uint8_t *)L.host_w[r];
        b.dst[r] = (uint8_t *)L.dev_region[r];
        b.vec[r] = r < L.n_regions ? L.region_bytes[r] / 16 : 0;
        b.per_job += b.vec[r];
    }
    stream_experts_kernel<<<4 * L.num_sms, 256, 0, s>>>(b);
    return 2;
}

// moe_get_residency
moe_status residency_read(Layer &L, int32_t *expert_of, int64_t *stats)
{
    if (L.S <= 0) return res_fail(MOE_ERR_UNSUPPORTED, "the layer keeps every expert resident");
    if (cudaDeviceSynchronize() != cudaSuccess) return res_fail(MOE_ERR_CUDA, "synchronize");
    if (expert_of && cudaMemcpy(expert_of, L.expert_of, (size_t)L.S * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return res_fail(MOE_ERR_CUDA, "read the slot table");
    if (stats) {
        unsigned long long st[4];
        if (cudaMemcpy(st, L.res_stats, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
            return res_fail(MOE_ERR_CUDA, "read the counters");
        for (int i = 0; i < 3; ++i) stats[i] = (int64_t)st[i];
    }
    return MOE_OK;
}

}  // namespace moe
