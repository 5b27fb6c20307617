// art_api.cu -- host side of libart: argument checks, the plan kernel, and the
// C entry points declared in include/art.h.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <cstddef>
#include <string>

#include "art_units.cuh"

namespace art {

template <bool kBF16, int D, int G, bool kART>
cudaError_t launch_main(Params p, cudaStream_t stream, int force_stages, LaunchInfo* li);

// The kernels are compiled in their own translation units (art_inst_*.cu,
// art_units_d*.cu); here they are only called.
#define ART_EXTERN_MAIN(BF, D, G)                                                                      \
    extern template cudaError_t launch_main<BF, D, G, true>(Params, cudaStream_t, int, LaunchInfo*); \
    extern template cudaError_t launch_main<BF, D, G, false>(Params, cudaStream_t, int, LaunchInfo*);
#define ART_EXTERN_UNITS(D, G)                                                                        \
    extern template cudaError_t launch_units<D, G, true>(Params, UParams, cudaStream_t, LaunchInfo*); \
    extern template cudaError_t launch_units<D, G, false>(Params, UParams, cudaStream_t, LaunchInfo*);
#define ART_EXTERN_ALL_G(M, ...) M(__VA_ARGS__, 1) M(__VA_ARGS__, 2) M(__VA_ARGS__, 4) M(__VA_ARGS__, 7) M(__VA_ARGS__, 8)
ART_EXTERN_ALL_G(ART_EXTERN_MAIN, true, 128)
ART_EXTERN_ALL_G(ART_EXTERN_MAIN, true, 64)
ART_EXTERN_ALL_G(ART_EXTERN_MAIN, false, 128)
ART_EXTERN_ALL_G(ART_EXTERN_MAIN, false, 64)
ART_EXTERN_ALL_G(ART_EXTERN_UNITS, 128)
ART_EXTERN_ALL_G(ART_EXTERN_UNITS, 64)
#undef ART_EXTERN_ALL_G
#undef ART_EXTERN_UNITS
#undef ART_EXTERN_MAIN

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
    // unit path (units != 0): its per-item and per-unit state, and the unit list;
    // ctas = CTAs of the unit kernel (sets the unit length), patience = the call's;
    // dense = the full-scan twin (every item stops at its last block, no fix pieces)
    int units, maxk, ctas, patience, dense;
    int ck_force;  // unit length forced by ART_CK (0: chosen here)
    int* p0;
    int* stop_min;
    int* resolved;
    int* fail;
    int* tflag;
    int* uflags;
    int2* ulist;
};

// Exclusive prefix sum of one value per thread over the CTA's kPlanThreads
// threads (warp shuffles, then the warp totals); `total` receives the sum.
// `s_warp` holds kPlanThreads / 32 words of shared memory.
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* s_warp, long long& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
        long long t = lane < kPlanThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kPlanThreads / 32) s_warp[lane] = t;  // inclusive warp totals
    }
    __syncthreads();
    total = s_warp[kPlanThreads / 32 - 1];
    const long long before = w > 0 ? s_warp[w - 1] : 0;
    __syncthreads();  // s_warp may be reused by the caller right away
    return before + x - v;
}

// One CTA per item: count the visit list (up to the first -1), check every
// listed block and its pages, and record n and flags. The last CTA to finish
// writes the claim order: items by visit-list length, longest first.
// Unit path: each CTA also clears its item's unit state and records the list
// position of block 0. The last CTA picks the unit length ck (8..16 blocks, at
// least the patience) so that the units fill whole waves of the unit kernel's
// CTAs, orders the items by units, and numbers the units round by round: unit
// k of the items that have one, in claim order, then unit k + 1 (ck fix pieces
// per item follow).
__global__ void __launch_bounds__(kPlanThreads) art_plan_kernel(const PlanParams p) {
    __shared__ unsigned int bitmap[kBitmapWords];
    __shared__ int s_hist[kSortBuckets];
    __shared__ long long s_warp[kPlanThreads / 32];
    __shared__ int s_n, s_flags, s_last, s_p0;
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
        s_p0 = 0x7fffffff;
    }
    __syncthreads();
    if (vrow) {
        // the first -1: a minimum per thread, per warp, then one shared atomic per warp
        int first_end = 0x7fffffff;
        for (int pos = tid; pos < p.max_visit; pos += kPlanThreads)
            if (vrow[pos] == -1) first_end = min(first_end, pos);
        first_end = __reduce_min_sync(0xffffffffu, first_end);
        if ((tid & 31) == 0 && first_end != 0x7fffffff) atomicMin(&s_n, first_end);
    }
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
        if (c == 0) {
            has0 = 1;
            atomicMin(&s_p0, pos);
        }
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
    if (p.units)
        for (int k = tid; k < p.maxk; k += kPlanThreads) {
            const size_t iu = (size_t)item * p.maxk + k;
            p.tflag[iu] = 0;
            reinterpret_cast<int4*>(p.uflags)[iu] = make_int4(0, 0, 0, 0);
        }
    __syncthreads();
    if (tid == 0) {
        const int e = s_flags >> 8;
        ItemInfo inf;
        inf.n = n;
        inf.flags = (s_flags & kItemHas0) | (e ? kItemBad : 0);
        p.info[item] = inf;
        if (p.units) {
            p.p0[item] = (s_flags & kItemHas0) ? s_p0 : -1;
            p.stop_min[item] = 0x7fffffff;
            p.resolved[item] = 0;
            p.fail[item] = 0;
        }
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
    // unit path: the unit length. With the lists' blocks spread over `ctas` CTAs in
    // w waves of at most 16 blocks each, ck = total / (w ctas) rounded up, in 8..16
    // and at least the patience (the count entering a unit then depends on the
    // previous unit only)
    __shared__ int s_ck;
    if (p.units) {
        int part = 0;
        for (int it = tid; it < p.num_items; it += kPlanThreads) {
            const int2 v = __ldcg(reinterpret_cast<const int2*>(&p.info[it]));
            part += (v.y & kItemBad) ? 0 : v.x;
        }
        long long total = 0;
        (void)block_exclusive_scan(part, s_warp, total);
        if (tid == 0) {
            const long long cap = (long long)kUnitBlocks * p.ctas;
            const long long waves = total > 0 ? (total + cap - 1) / cap : 1;
            long long ck = (total + waves * p.ctas - 1) / (waves * p.ctas);
            ck = ck < kUnitMinBlocks ? kUnitMinBlocks : ck > kUnitBlocks ? kUnitBlocks : ck;
            if (p.ck_force) ck = p.ck_force;
            if (ck < p.patience) ck = p.patience;
            s_ck = (int)ck;
            p.hdr->ck = (int)ck;
        }
        __syncthreads();
    }
    // sort key: the list length, or (unit path) the units of the list
    auto sort_key = [&](int it) -> int {
        const int2 v = __ldcg(reinterpret_cast<const int2*>(&p.info[it]));
        if (!p.units) return v.x;
        return (v.y & kItemBad) ? 0 : (v.x + s_ck - 1) / s_ck;
    };
    for (int it = tid; it < p.num_items; it += kPlanThreads) {
        const int nn = sort_key(it);
        atomicAdd(&s_hist[kSortBuckets - 1 - min(nn, kSortBuckets - 1)], 1);
    }
    __syncthreads();
    constexpr int per = kSortBuckets / kPlanThreads;
    int sum = 0;
    for (int i = 0; i < per; ++i) sum += s_hist[tid * per + i];
    long long all_items = 0;
    int run = (int)block_exclusive_scan(sum, s_warp, all_items);
    for (int i = 0; i < per; ++i) {
        const int t = s_hist[tid * per + i];
        s_hist[tid * per + i] = run;
        run += t;
    }
    __syncthreads();
    for (int it = tid; it < p.num_items; it += kPlanThreads) {
        const int nn = sort_key(it);
        const int pos = atomicAdd(&s_hist[kSortBuckets - 1 - min(nn, kSortBuckets - 1)], 1);
        p.order[pos] = it;
    }
    if (!p.units) return;
    // unit path: cnt_k = items with more than k units (a prefix of the claim order, which
    // is by units, descending), S_k = units numbered before round k; unit k of the item
    // at claim position o gets number S_k + o
    __syncthreads();
    for (int i = tid; i < kSortBuckets; i += kPlanThreads) s_hist[i] = 0;
    __syncthreads();
    for (int it = tid; it < p.num_items; it += kPlanThreads) {
        const int nn = sort_key(it);  // <= maxk < kUnitMaxK = kSortBuckets
        if (nn > 0) atomicAdd(&s_hist[nn - 1], 1);
    }
    __syncthreads();
    // items with at most k units = exclusive prefix P_k of the histogram; cnt_k = items - P_k
    {
        int csum = 0;
        for (int i = 0; i < per; ++i) csum += s_hist[tid * per + i];
        long long tot = 0;
        int run2 = (int)block_exclusive_scan(csum, s_warp, tot);
        const int with_units = (int)tot;
        for (int i = 0; i < per; ++i) {
            const int k = tid * per + i;
            const int hk = s_hist[k];
            s_hist[k] = with_units - run2;  // cnt_k
            run2 += hk;
        }
    }
    __syncthreads();
    {
        int csum = 0;
        for (int i = 0; i < per; ++i) csum += s_hist[tid * per + i];
        long long n_reg = 0;
        int acc = (int)block_exclusive_scan(csum, s_warp, n_reg);
        if (tid == 0) {
            p.hdr->n_regular = (int)n_reg;
            p.hdr->n_units = (int)n_reg + (p.dense ? 0 : p.num_items * s_ck);  // then ck fix pieces per item
        }
        for (int i = 0; i < per; ++i) {
            const int k = tid * per + i;
            const int t = s_hist[k];
            s_hist[k] = acc;  // S_k
            acc += t;
        }
    }
    __syncthreads();
    for (int o = tid; o < p.num_items; o += kPlanThreads) {
        const int my_item = __ldcg(&p.order[o]);
        const int my_nch = sort_key(my_item);
        for (int k = 0; k < my_nch; ++k) p.ulist[s_hist[k] + o] = make_int2(my_item, k);
        if (p.dense && my_nch > 0) {
            // the twin reads every listed block: each item stops at its last one
            p.stop_min[my_item] = __ldcg(reinterpret_cast<const int*>(&p.info[my_item])) - 1;
            p.resolved[my_item] = my_nch;
        }
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

template <int D, int G, bool kART>
cudaError_t launch_units(Params p, UParams up, cudaStream_t stream, LaunchInfo* li);

template <bool kART>
static cudaError_t dispatch_units(const art_shape& s, const Params& p, const UParams& up, cudaStream_t st,
                                  LaunchInfo* li) {
    const int G = s.num_q_heads / s.num_kv_heads;
#define ART_UCASE(DD, GG) \
    if (s.head_dim == DD && G == GG) return launch_units<DD, GG, kART>(p, up, st, li);
#define ART_UCASES(DD) ART_UCASE(DD, 1) ART_UCASE(DD, 2) ART_UCASE(DD, 4) ART_UCASE(DD, 7) ART_UCASE(DD, 8)
    ART_UCASES(128)
    ART_UCASES(64)
#undef ART_UCASES
#undef ART_UCASE
    return cudaErrorInvalidValue;
}

// The unit path (one item spread over many CTAs) is offered for bf16 when its
// workspace area, sized for the longest list the block table allows, stays within
// kUnitMaxWsBytes.
static int unit_maxk(const art_shape& s) {
    const long long tmax = ((long long)s.max_pages_per_seq * s.page_size + kBK - 1) / kBK;
    const long long k = (tmax + kUnitMinBlocks - 1) / kUnitMinBlocks;
    return k > kUnitMaxK ? 0 : (int)k;
}

static size_t unit_bytes(const art_shape& s) {
    const int items = s.batch * s.num_kv_heads;
    return make_unit_ws(items, unit_maxk(s), s.head_dim, s.num_q_heads / s.num_kv_heads).total;
}

static bool unit_eligible(const art_shape& s) {
    return s.dtype == ART_DTYPE_BF16 && unit_maxk(s) >= 1 && unit_maxk(s) < kUnitMaxK &&
           unit_bytes(s) <= kUnitMaxWsBytes;
}

static size_t unit_area_offset(int num_items) { return align_up(workspace_bytes_for(num_items), 256); }

// Unit path or one CTA per item: ART_UNITS=0/1 forces the choice (where the
// path is offered). Otherwise ART takes the unit path when there are fewer items
// than half the SMs, and the dense twin when there are fewer items than SMs (its
// full scan has no stop to find). Measured for the full scan: 128 items on 152
// SMs 0.359 ms on units against 0.375 ms; with more items one CTA per SM is as
// fast or faster (ragged batch 1.288 against 1.303 ms, paged 0.665 against 0.703).
static bool want_units(const art_shape& s, int patience, size_t workspace_bytes, bool dense = false) {
    if (!unit_eligible(s) || (!dense && (patience > kUnitBlocks || s.num_probe > kMaxProbe))) return false;
    const int items = s.batch * s.num_kv_heads;
    if (workspace_bytes < unit_area_offset(items) + unit_bytes(s)) return false;
    const char* env = std::getenv("ART_UNITS");
    if (env) return std::atoi(env) != 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    // the full scan: units while some SM would get no item (with more items, one CTA
    // per SM streams as fast or faster); ART: units below half the SMs (its
    // statistics cost more per block on the unit path)
    return dense ? items < sms : 2 * items < sms;
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
        // more than kMaxProbe probe columns per head: bf16 only (one CTA per item)
        if (s.num_probe > kMaxProbe && s.dtype != ART_DTYPE_BF16) return ART_ERR_UNSUPPORTED;
        if (patience < 1) return ART_ERR_INVALID_ARG;
        if (std::isnan(eps_mag) || std::isnan(eps_dir) || eps_mag < 0.f || eps_dir < 0.f) return ART_ERR_INVALID_ARG;
    }
    const int num_items = s.batch * s.num_kv_heads;
    if (workspace_bytes < workspace_bytes_for(num_items)) return ART_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = static_cast<WsHeader*>(workspace);
    ItemInfo* info = reinterpret_cast<ItemInfo*>(hdr + 1);
    int32_t* order = reinterpret_cast<int32_t*>(info + num_items);

    const bool units = want_units(s, kART ? patience : 1, workspace_bytes, !kART);
    UParams up;
    std::memset(&up, 0, sizeof up);
    if (units) {
        unsigned char* base = static_cast<unsigned char*>(workspace) + unit_area_offset(num_items);
        const UnitWs w = make_unit_ws(num_items, unit_maxk(s), s.head_dim, s.num_q_heads / s.num_kv_heads);
        up.ulist = reinterpret_cast<const int2*>(base + w.ulist);
        up.p0 = reinterpret_cast<const int*>(base + w.p0);
        up.stop_min = reinterpret_cast<int*>(base + w.stop_min);
        up.resolved = reinterpret_cast<int*>(base + w.resolved);
        up.fail = reinterpret_cast<int*>(base + w.fail);
        up.tflag = reinterpret_cast<int*>(base + w.tflag);
        up.uflags = reinterpret_cast<int*>(base + w.uflags);
        up.agg = reinterpret_cast<float*>(base + w.agg);
        up.incl = reinterpret_cast<float*>(base + w.incl);
        up.part_o = reinterpret_cast<float*>(base + w.part_o);
        up.part_ml = reinterpret_cast<float*>(base + w.part_ml);
        up.fix_o = reinterpret_cast<float*>(base + w.fix_o);
        up.fix_ml = reinterpret_cast<float*>(base + w.fix_ml);
        up.ustore = reinterpret_cast<float*>(base + w.ustore);
        up.ck = 0;  // chosen on the device by the plan kernel
        up.maxk = unit_maxk(s);
    }

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
    pp.units = units ? 1 : 0;
    pp.maxk = up.maxk;
    pp.patience = kART ? patience : 1;
    pp.dense = kART ? 0 : 1;
    pp.ctas = 0;
    pp.ck_force = 0;
    if (const char* eck = std::getenv("ART_CK")) {
        const int v = std::atoi(eck);
        if (v >= kUnitMinBlocks && v <= kUnitBlocks) pp.ck_force = v;
    }
    if (units) {
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        pp.ctas = 2 * sms;  // the unit kernel runs two CTAs per SM
    }
    pp.p0 = const_cast<int*>(up.p0);
    pp.stop_min = up.stop_min;
    pp.resolved = up.resolved;
    pp.fail = up.fail;
    pp.tflag = up.tflag;
    pp.uflags = up.uflags;
    pp.ulist = const_cast<int2*>(up.ulist);
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
    // ART_TEST_STALL_NS=<ns> (tests of the failure path only): the consumer warps wait
    // on a barrier that nothing completes, and every bounded wait gives up after <ns>
    p.wait_ns = kWaitLimitNs;
    p.stall = 0;
    if (const char* es = std::getenv("ART_TEST_STALL_NS")) {
        const long long ns = std::atoll(es);
        if (ns > 0) {
            p.stall = 1;
            p.wait_ns = (unsigned long long)(ns < (long long)kWaitLimitNs ? ns : (long long)kWaitLimitNs);
        }
    }
    if (t_events.start && (e = cudaEventRecord(t_events.start, st)) != cudaSuccess) return cuda_fail(e);
    e = units ? dispatch_units<kART>(s, p, up, st, li) : dispatch<kART>(s, p, st, env_stages(), li);
    if (e != cudaSuccess) return cuda_fail(e);
    if (t_events.stop && (e = cudaEventRecord(t_events.stop, st)) != cudaSuccess) return cuda_fail(e);
    return ART_OK;
}

}  // namespace art

using namespace art;

extern "C" {

size_t art_workspace_bytes(const art_shape* shape) {
    if (!shape || shape->batch < 1 || shape->num_kv_heads < 1) return 0;
    const int items = shape->batch * shape->num_kv_heads;
    if (check_shape(shape) == ART_OK && unit_eligible(*shape)) return unit_area_offset(items) + unit_bytes(*shape);
    return workspace_bytes_for(items);
}

int art_decode_path(const art_shape* shape, int32_t patience, size_t workspace_bytes) {
    if (check_shape(shape) != ART_OK) return 0;
    return want_units(*shape, patience, workspace_bytes) ? 1 : 0;
}

int dense_decode_path(const art_shape* shape, size_t workspace_bytes) {
    if (check_shape(shape) != ART_OK) return 0;
    return want_units(*shape, 1, workspace_bytes, true) ? 1 : 0;
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

// Device address of g_static_workspace on the current device, looked up on every
// call: the lookup allocates nothing, and an address kept from an earlier call could
// be stale after the device's context was reset and the module loaded again.
static int static_workspace(void** out) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!ptr) return ART_ERR_LAUNCH;
    *out = ptr;
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

extern "C" int art_read_static_status(int32_t* status) {
    if (!status) return ART_ERR_INVALID_ARG;
    const cudaError_t e =
        cudaMemcpyFromSymbol(status, art::g_static_workspace, sizeof(int32_t), offsetof(art::WsHeader, status));
    if (e != cudaSuccess) return cuda_fail(e);
    return ART_OK;
}
