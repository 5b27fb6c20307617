// art_api.cu -- host side of libart: argument checks, the plan kernel, and the
// C entry points declared in include/art.h.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "art_common.cuh"

namespace art {

template <bool kBF16, int D, int G, bool kART>
cudaError_t launch_main(Params p, cudaStream_t stream, int force_stages, LaunchInfo* li);

constexpr int kPlanThreads = 256;
constexpr int kBitmapWords = 2048;  // duplicate detection for lists over up to 65536 blocks
constexpr int kSortBuckets = 4096;  // LPT bucketing of visit-list lengths

struct PlanParams {
    const int32_t* seq_lens;
    const int32_t* visit;
    const int32_t* block_table;
    const int32_t* probe;  // checked when non-null
    WsHeader* hdr;
    int32_t* order;
    ItemInfo* info;
    int Hkv, Ps, max_pages, max_visit, m, D, num_pages, num_items;
};

// One CTA per item: count the visit list (up to the first -1), check every
// listed block and its pages, and record n and flags. The last CTA to finish
// writes the claim order: items by visit-list length, longest first.
__global__ void __launch_bounds__(kPlanThreads) art_plan_kernel(const PlanParams p) {
    __shared__ unsigned int bitmap[kBitmapWords];
    __shared__ int s_hist[kSortBuckets];
    __shared__ int s_part[kPlanThreads];
    __shared__ int s_n, s_flags, s_last;
    const int item = blockIdx.x, tid = threadIdx.x;
    const int b = item / p.Hkv;
    const int seq_len = p.seq_lens[b];
    const bool seq_ok = seq_len >= 0 && (long long)seq_len <= (long long)p.max_pages * p.Ps;
    const int T = seq_ok ? (seq_len + kBK - 1) / kBK : 0;
    const bool dupcheck = T <= kBitmapWords * 32;
    const int32_t* vrow = p.visit ? p.visit + (size_t)item * p.max_visit : nullptr;
    const int32_t* trow = p.block_table + (size_t)b * p.max_pages;
    for (int i = tid; i < kBitmapWords; i += kPlanThreads) bitmap[i] = 0;
    if (tid == 0) {
        s_n = vrow ? p.max_visit : T;
        s_flags = 0;
    }
    __syncthreads();
    if (vrow)
        for (int pos = tid; pos < p.max_visit; pos += kPlanThreads)
            if (vrow[pos] == -1) atomicMin(&s_n, pos);
    __syncthreads();
    const int n = seq_ok ? s_n : 0;
    int err = seq_ok ? 0 : ART_STATUS_BAD_SEQLEN;
    int has0 = 0;
    for (int pos = tid; pos < n; pos += kPlanThreads) {
        const int c = vrow ? vrow[pos] : pos;
        if (c < 0 || c >= T) {
            err |= ART_STATUS_BAD_VISIT;
            continue;
        }
        if (c == 0) has0 = 1;
        if (dupcheck) {
            const unsigned int bit = 1u << (c & 31);
            if (atomicOr(&bitmap[c >> 5], bit) & bit) err |= ART_STATUS_DUP_VISIT;
        }
        const int t0 = c * kBK;
        const int nv = min(kBK, seq_len - t0);
        if (p.Ps <= kBK) {
            const int npv = (nv + p.Ps - 1) / p.Ps, first = t0 / p.Ps;
            for (int k = 0; k < npv; ++k) {
                const int pg = trow[first + k];
                if (pg < 0 || pg >= p.num_pages) err |= ART_STATUS_BAD_PAGE;
            }
        } else {
            const int pg = trow[t0 / p.Ps];
            if (pg < 0 || pg >= p.num_pages) err |= ART_STATUS_BAD_PAGE;
        }
    }
    if (p.probe && tid < p.m) {
        const int col = p.probe[tid];
        if (col < 0 || col >= p.D) err |= ART_STATUS_BAD_PROBE;
        for (int k = 0; k < p.m; ++k)
            if (k != tid && p.probe[k] == col) err |= ART_STATUS_BAD_PROBE;
    }
    if (has0) atomicOr(&s_flags, kItemHas0);
    if (err) atomicOr(&s_flags, err << 8);
    __syncthreads();
    if (tid == 0) {
        const int e = s_flags >> 8;
        ItemInfo inf;
        inf.n = n;
        inf.flags = (s_flags & kItemHas0) | (e ? kItemBad : 0);
        p.info[item] = inf;
        if (e) atomicOr(&p.hdr->status, e);
        __threadfence();
        s_last = (atomicAdd(&p.hdr->plan_done, 1u) == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // counting sort of the items by n, descending (buckets of n clamped at 4095)
    for (int i = tid; i < kSortBuckets; i += kPlanThreads) s_hist[i] = 0;
    __syncthreads();
    for (int it = tid; it < p.num_items; it += kPlanThreads) {
        const int nn = __ldcg(reinterpret_cast<const int*>(&p.info[it]));
        atomicAdd(&s_hist[kSortBuckets - 1 - min(nn, kSortBuckets - 1)], 1);
    }
    __syncthreads();
    constexpr int per = kSortBuckets / kPlanThreads;
    int sum = 0;
    for (int i = 0; i < per; ++i) sum += s_hist[tid * per + i];
    s_part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int i = 0; i < kPlanThreads; ++i) {
            const int t = s_part[i];
            s_part[i] = run;
            run += t;
        }
    }
    __syncthreads();
    int run = s_part[tid];
    for (int i = 0; i < per; ++i) {
        const int t = s_hist[tid * per + i];
        s_hist[tid * per + i] = run;
        run += t;
    }
    __syncthreads();
    for (int it = tid; it < p.num_items; it += kPlanThreads) {
        const int nn = __ldcg(reinterpret_cast<const int*>(&p.info[it]));
        const int pos = atomicAdd(&s_hist[kSortBuckets - 1 - min(nn, kSortBuckets - 1)], 1);
        p.order[pos] = it;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
thread_local std::string g_last_cuda_error = "no error";

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = cudaGetErrorString(e);
    return ART_ERR_LAUNCH;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

static int check_shape(const art_shape* s) {
    if (!s) return ART_ERR_INVALID_ARG;
    if (s->batch < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 || s->head_dim < 1 || s->page_size < 1 ||
        s->block_size < 1 || s->max_pages_per_seq < 1 || s->max_visit < 1 || s->num_pages_total < 1)
        return ART_ERR_INVALID_ARG;
    if (s->num_q_heads % s->num_kv_heads != 0) return ART_ERR_INVALID_ARG;
    if (s->dtype != ART_DTYPE_BF16 && s->dtype != ART_DTYPE_F32) return ART_ERR_INVALID_ARG;
    if ((long long)s->batch * s->num_kv_heads > (1LL << 30)) return ART_ERR_UNSUPPORTED;
    const int G = s->num_q_heads / s->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 7 && G != 8) return ART_ERR_UNSUPPORTED;
    if (s->head_dim != 64 && s->head_dim != 128) return ART_ERR_UNSUPPORTED;
    if (s->block_size != kBK) return ART_ERR_UNSUPPORTED;
    if (!pow2(s->page_size) || s->page_size < 8 || s->page_size > 4096) return ART_ERR_UNSUPPORTED;
    return ART_OK;
}

template <bool kART>
static cudaError_t dispatch(const art_shape& s, const Params& p, cudaStream_t st, int force_stages,
                            LaunchInfo* li) {
    const int G = s.num_q_heads / s.num_kv_heads;
    const bool bf = s.dtype == ART_DTYPE_BF16;
#define ART_CASE(BF, DD, GG)                                 \
    if (bf == BF && s.head_dim == DD && G == GG)             \
        return launch_main<BF, DD, GG, kART>(p, st, force_stages, li);
#define ART_CASES(BF, DD) ART_CASE(BF, DD, 1) ART_CASE(BF, DD, 2) ART_CASE(BF, DD, 4) ART_CASE(BF, DD, 7) ART_CASE(BF, DD, 8)
    ART_CASES(true, 128)
    ART_CASES(true, 64)
    ART_CASES(false, 64)
    ART_CASES(false, 128)
#undef ART_CASES
#undef ART_CASE
    return cudaErrorInvalidValue;
}

// events recorded around the decode-kernel launch of this thread's calls
struct TimingEvents {
    cudaEvent_t start = nullptr, stop = nullptr;
};
static thread_local TimingEvents t_events;

static int env_stages() {
    const char* e = std::getenv("ART_STAGES");
    return e ? std::atoi(e) : 0;
}

template <bool kART>
static int run(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
               const int32_t* seq_lens, const int32_t* visit_order, float eps_mag, float eps_dir, int32_t patience,
               const int32_t* probe_idx, void* out, int32_t* blocks_used, const art_shape* shape, void* workspace,
               size_t workspace_bytes, void* stream, LaunchInfo* li, int probe_heads = 0) {
    const int rc = check_shape(shape);
    if (rc != ART_OK) return rc;
    const art_shape& s = *shape;
    if (probe_heads < 0 || probe_heads > s.num_q_heads / s.num_kv_heads) return ART_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace) return ART_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
        return ART_ERR_INVALID_ARG;
    if (kART) {
        if (!probe_idx || !blocks_used) return ART_ERR_INVALID_ARG;
        if (s.num_probe < 1 || s.num_probe > s.head_dim) return ART_ERR_INVALID_ARG;
        if (s.num_probe > kMaxProbe) return ART_ERR_UNSUPPORTED;
        if (patience < 1) return ART_ERR_INVALID_ARG;
        if (std::isnan(eps_mag) || std::isnan(eps_dir) || eps_mag < 0.f || eps_dir < 0.f) return ART_ERR_INVALID_ARG;
    }
    const int num_items = s.batch * s.num_kv_heads;
    if (workspace_bytes < workspace_bytes_for(num_items)) return ART_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = static_cast<WsHeader*>(workspace);
    ItemInfo* info = reinterpret_cast<ItemInfo*>(hdr + 1);
    int32_t* order = reinterpret_cast<int32_t*>(info + num_items);

    cudaError_t e = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st);
    if (e != cudaSuccess) return cuda_fail(e);
    PlanParams pp;
    pp.seq_lens = seq_lens;
    pp.visit = visit_order;
    pp.block_table = block_table;
    pp.probe = kART ? probe_idx : nullptr;
    pp.hdr = hdr;
    pp.order = order;
    pp.info = info;
    pp.Hkv = s.num_kv_heads;
    pp.Ps = s.page_size;
    pp.max_pages = s.max_pages_per_seq;
    pp.max_visit = s.max_visit;
    pp.m = kART ? s.num_probe : 0;
    pp.D = s.head_dim;
    pp.num_pages = s.num_pages_total;
    pp.num_items = num_items;
    art_plan_kernel<<<num_items, kPlanThreads, 0, st>>>(pp);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);

    Params p;
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.visit = visit_order;
    p.probe = kART ? probe_idx : nullptr;
    p.out = out;
    p.blocks_used = kART ? blocks_used : nullptr;
    p.hdr = hdr;
    p.order = order;
    p.info = info;
    p.B = s.batch;
    p.Hq = s.num_q_heads;
    p.Hkv = s.num_kv_heads;
    p.Ps = s.page_size;
    p.max_pages = s.max_pages_per_seq;
    p.max_visit = s.max_visit;
    p.m = kART ? s.num_probe : 0;
    p.num_pages = s.num_pages_total;
    p.num_items = num_items;
    p.stages = 0;
    p.eps_mag = eps_mag;
    p.eps_dir = eps_dir;
    p.patience = patience;
    p.ph = probe_heads > 0 ? probe_heads : s.num_q_heads / s.num_kv_heads;
    p.tma3d = 0;
    if (t_events.start && (e = cudaEventRecord(t_events.start, st)) != cudaSuccess) return cuda_fail(e);
    e = dispatch<kART>(s, p, st, env_stages(), li);
    if (e != cudaSuccess) return cuda_fail(e);
    if (t_events.stop && (e = cudaEventRecord(t_events.stop, st)) != cudaSuccess) return cuda_fail(e);
    return ART_OK;
}

}  // namespace art

using namespace art;

extern "C" {

size_t art_workspace_bytes(const art_shape* shape) {
    if (!shape || shape->batch < 1 || shape->num_kv_heads < 1) return 0;
    return workspace_bytes_for(shape->batch * shape->num_kv_heads);
}

int art_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
               const int32_t* seq_lens, const int32_t* visit_order, float eps_mag, float eps_dir, int32_t patience,
               const int32_t* probe_idx, void* out, int32_t* blocks_used, const art_shape* shape, void* workspace,
               size_t workspace_bytes, void* stream) {
    return run<true>(q, k_cache, v_cache, block_table, seq_lens, visit_order, eps_mag, eps_dir, patience, probe_idx,
                     out, blocks_used, shape, workspace, workspace_bytes, stream, nullptr);
}

int art_decode_ex(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                  const int32_t* seq_lens, const int32_t* visit_order, float eps_mag, float eps_dir, int32_t patience,
                  const int32_t* probe_idx, void* out, int32_t* blocks_used, const art_shape* shape, void* workspace,
                  size_t workspace_bytes, void* stream, const art_options* options) {
    if (options) {
        for (int i = 0; i < 7; ++i)
            if (options->reserved[i] != 0) return ART_ERR_INVALID_ARG;
    }
    return run<true>(q, k_cache, v_cache, block_table, seq_lens, visit_order, eps_mag, eps_dir, patience, probe_idx,
                     out, blocks_used, shape, workspace, workspace_bytes, stream, nullptr,
                     options ? options->probe_heads : 0);
}

int dense_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                 const int32_t* seq_lens, const int32_t* visit_order, void* out, const art_shape* shape,
                 void* workspace, size_t workspace_bytes, void* stream) {
    return run<false>(q, k_cache, v_cache, block_table, seq_lens, visit_order, 0.f, 0.f, 1, nullptr, out, nullptr,
                      shape, workspace, workspace_bytes, stream, nullptr);
}

int art_read_device_status(const void* workspace, int32_t* status) {
    if (!workspace || !status) return ART_ERR_INVALID_ARG;
    const WsHeader* hdr = static_cast<const WsHeader*>(workspace);
    cudaError_t e = cudaMemcpy(status, &hdr->status, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return ART_OK;
}

const char* art_status_string(int code) {
    switch (code) {
        case ART_OK: return "ok";
        case ART_ERR_INVALID_ARG: return "invalid argument";
        case ART_ERR_UNSUPPORTED: return "unsupported size";
        case ART_ERR_WORKSPACE: return "workspace too small";
        case ART_ERR_LAUNCH: return "CUDA launch or call failed";
        default: return "unknown code";
    }
}

const char* art_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

void art_set_timing_events(void* start, void* stop) {
    t_events.start = static_cast<cudaEvent_t>(start);
    t_events.stop = static_cast<cudaEvent_t>(stop);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// art_decode_static: art_decode with its workspace in a device array that
// lives inside this library, for callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace art {

constexpr int kStaticMaxItems = 16384;  // largest batch * num_kv_heads accepted
constexpr size_t kStaticWorkspaceBytes =
    (sizeof(WsHeader) + (size_t)kStaticMaxItems * (sizeof(int32_t) + sizeof(ItemInfo)) + 255) / 256 * 256;

// One copy per device that loads this library, kept until the process exits.
// In host code this name only stands for the device array; its device address
// comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kStaticMaxDevices = 256;
static void* g_static_workspace_addr[kStaticMaxDevices];
static std::mutex g_static_mutex;

// Device address of g_static_workspace on the current device; looked up once
// per device, on that device's first call.
static int static_workspace(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kStaticMaxDevices) return ART_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_workspace_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_workspace);
        if (e != cudaSuccess) return cuda_fail(e);
        if (!ptr) return ART_ERR_LAUNCH;
        g_static_workspace_addr[dev] = ptr;
    }
    *out = g_static_workspace_addr[dev];
    return ART_OK;
}

}  // namespace art

extern "C" int art_decode_static(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                 const int32_t* seq_lens, const int32_t* visit_order, float eps_mag, float eps_dir,
                                 int32_t patience, const int32_t* probe_idx, void* out, int32_t* blocks_used,
                                 const art_shape* shape, void* stream) {
    const int rc = check_shape(shape);
    if (rc != ART_OK) return rc;
    if ((long long)shape->batch * shape->num_kv_heads > kStaticMaxItems) return ART_ERR_UNSUPPORTED;
    void* ws = nullptr;
    const int rs = static_workspace(&ws);
    if (rs != ART_OK) return rs;
    return run<true>(q, k_cache, v_cache, block_table, seq_lens, visit_order, eps_mag, eps_dir, patience, probe_idx,
                     out, blocks_used, shape, ws, kStaticWorkspaceBytes, stream, nullptr);
}
