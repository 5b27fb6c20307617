// art_select.cu -- key-based block selection that writes an ART visit list.
//
// A KV manager that keeps only the blocks whose keys score high for the
// current queries hands ART a short list; ART then stops early inside that
// list (ART paper sec. 4: composition with key-centric KV selection). The
// score of block c of item (b, g) is the pooled estimate of FlexPrefill's
// block selection (FlexPrefill summary, pooled block scores):
//     score_c = mean_{h in group g}(q_h) . mean_{t in block c}(k_t)
// over the tokens of the block below seq_len. Kept: the ceil(top_frac * T)
// highest scores (equal scores: the lower block index first), block 0 (the
// attention sink) and the last keep_last blocks. Written order: block 0, then
// the other kept blocks by descending index (most recent first) or, on request,
// by descending score (importance first), then -1.
//
// Two kernels: art_score_kernel (many CTAs per item, each scoring a run of
// blocks; bound by reading K once) and art_topk_kernel (one CTA per item: a
// bitonic sort of the item's scores in shared memory, then the list).
#include <cmath>

#include "art_common.cuh"

namespace art {

constexpr int kScoreThreads = 256;      // 8 warps, one block at a time each
constexpr int kScoreBlocksPerCta = 16;  // blocks scored by one CTA
constexpr int kTopkThreads = 1024;
constexpr int kMaxSelectBlocks = 8192;  // blocks of one sequence (512k tokens)

struct SelectParams {
    const void* q;
    const void* k;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* scores;   // [num_items][maxT]
    int32_t* visit;  // [num_items][max_visit]
    WsHeader* hdr;
    int B, Hq, Hkv, Ps, max_pages, max_visit, num_pages, maxT, keep_last;
    int by_score;  // list order: 0 descending index, 1 descending score
    float top_frac;
};

template <bool kBF16>
__device__ __forceinline__ float load_elem(const void* base, size_t i) {
    if constexpr (kBF16) {
        const uint16_t b = static_cast<const uint16_t*>(base)[i];
        return __uint_as_float((uint32_t)b << 16);
    } else {
        return static_cast<const float*>(base)[i];
    }
}

// grid (ceil(maxT / kScoreBlocksPerCta), items): scores of blocks
// [x * kScoreBlocksPerCta, (x + 1) * kScoreBlocksPerCta) of item y.
template <bool kBF16, int D>
__global__ void __launch_bounds__(kScoreThreads) art_score_kernel(const SelectParams p) {
    constexpr int ELT = kBF16 ? 2 : 4;
    constexpr int CPR = D * ELT / 16;  // 16-byte chunks of a row
    constexpr int RPS = 32 / CPR;      // rows per warp step
    constexpr int EPC = 16 / ELT;      // elements per chunk
    constexpr int UNR = 8;             // row steps in flight per lane
    __shared__ float qbar[D];
    const int item = blockIdx.y;
    const int b = item / p.Hkv, g = item - (item / p.Hkv) * p.Hkv;
    const int G = p.Hq / p.Hkv;
    const int seq_len = p.seq_lens[b];
    if (seq_len < 0 || (long long)seq_len > (long long)p.max_pages * p.Ps) return;  // flagged by art_topk_kernel
    const int T = (seq_len + kBK - 1) / kBK;
    const int c0 = blockIdx.x * kScoreBlocksPerCta;
    if (c0 >= T) return;
    for (int col = threadIdx.x; col < D; col += kScoreThreads) {
        float s = 0.f;
        for (int h = 0; h < G; ++h) s += load_elem<kBF16>(p.q, ((size_t)b * p.Hq + (size_t)g * G + h) * D + col);
        qbar[col] = s / (float)G;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ch = lane % CPR, rsub = lane / CPR;
    float qv[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) qv[e] = qbar[ch * EPC + e];
    const int32_t* trow = p.block_table + (size_t)b * p.max_pages;
    const char* kb = static_cast<const char*>(p.k);
    const int PR = p.Ps < kBK ? p.Ps : kBK;  // rows of the block in one page
    for (int c = c0 + warp; c < min(c0 + kScoreBlocksPerCta, T); c += kScoreThreads / 32) {
        const int t0 = c * kBK, nv = min(kBK, seq_len - t0);
        // the block's pages (at most 8), one per lane, then shared by shuffles
        const int npg = (nv + PR - 1) / PR;
        int mypg = 0;
        if (lane < npg) mypg = __ldg(&trow[(t0 + lane * PR) / p.Ps]);
        const bool badpg = lane < npg && (mypg < 0 || mypg >= p.num_pages);
        bool bad = __any_sync(0xffffffffu, badpg);
        const int r_in = (t0 % p.Ps);  // first row of the block inside its page (pages longer than a block)
        float acc = 0.f;
        for (int r0 = 0; r0 < nv && !bad; r0 += RPS * UNR) {
            uint4 v[UNR];
            bool on[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int r = r0 + u * RPS + rsub;
                on[u] = r < nv;
                const int pg = __shfl_sync(0xffffffffu, mypg, on[u] ? r / PR : 0);
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (on[u]) {
                    const size_t row = ((size_t)pg * p.Hkv + g) * p.Ps + r_in + (r % PR);
                    v[u] = __ldg(reinterpret_cast<const uint4*>(kb + row * (D * ELT)) + ch);
                }
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                if (!on[u]) continue;
                const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                if constexpr (kBF16) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc = fmaf(__uint_as_float(w4[e] << 16), qv[2 * e], acc);
                        acc = fmaf(__uint_as_float(w4[e] & 0xffff0000u), qv[2 * e + 1], acc);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc = fmaf(__uint_as_float(w4[e]), qv[e], acc);
                }
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            if (bad) atomicOr(&p.hdr->status, ART_STATUS_BAD_PAGE);
            p.scores[(size_t)item * p.maxT + c] = bad ? __int_as_float(0x7fc00000) : acc / (float)nv;
        }
    }
}

// Before `a`/`b`: the higher score, then the lower block index; NaN sorts last.
__device__ __forceinline__ bool ranks_before(float sa, int ia, float sb, int ib) {
    const bool na = sa != sa, nb = sb != sb;
    if (na != nb) return nb;
    if (!na && sa != sb) return sa > sb;
    return ia < ib;
}

// One CTA per item: sort (score, index) pairs, mark the kept blocks, write the list.
__global__ void __launch_bounds__(kTopkThreads) art_topk_kernel(const SelectParams p) {
    extern __shared__ __align__(16) unsigned char sm[];
    float* key = reinterpret_cast<float*>(sm);                    // [N2]
    int* idx = reinterpret_cast<int*>(key + kMaxSelectBlocks);     // [N2]
    int* kept = idx + kMaxSelectBlocks;                            // [T] flags, then output positions
    __shared__ int s_wsum[kTopkThreads / 32];
    __shared__ int s_bad;
    const int item = blockIdx.x, tid = threadIdx.x;
    const int b = item / p.Hkv;
    const int seq_len = p.seq_lens[b];
    int32_t* out = p.visit + (size_t)item * p.max_visit;
    const bool seq_ok = seq_len >= 0 && (long long)seq_len <= (long long)p.max_pages * p.Ps;
    const int T = seq_ok ? (seq_len + kBK - 1) / kBK : 0;
    if (tid == 0) s_bad = seq_ok ? 0 : 1;
    __syncthreads();
    if (!seq_ok) {
        if (tid == 0) atomicOr(&p.hdr->status, ART_STATUS_BAD_SEQLEN);
        for (int i = tid; i < p.max_visit; i += kTopkThreads) out[i] = -1;
        return;
    }
    int N2 = 1;
    while (N2 < T) N2 <<= 1;
    for (int i = tid; i < N2; i += kTopkThreads) {
        const float s = i < T ? p.scores[(size_t)item * p.maxT + i] : -INFINITY;
        if (i < T && s != s) s_bad = 1;  // a bad page inside the item
        key[i] = i < T ? s : -INFINITY;
        idx[i] = i < T ? i : 0x7fffffff;
    }
    for (int i = tid; i < T; i += kTopkThreads) kept[i] = 0;
    __syncthreads();
    if (s_bad) {
        for (int i = tid; i < p.max_visit; i += kTopkThreads) out[i] = -1;
        return;
    }
    // bitonic sort into rank order
    for (int size = 2; size <= N2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < N2; i += kTopkThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;  // this run ends in rank order
                    const bool before = ranks_before(key[j], idx[j], key[i], idx[i]);
                    if (before == up) {
                        const float tk = key[i]; key[i] = key[j]; key[j] = tk;
                        const int ti = idx[i]; idx[i] = idx[j]; idx[j] = ti;
                    }
                }
            }
            __syncthreads();
        }
    }
    // kept: the top ceil(top_frac * T), block 0, the last keep_last
    const int ktop = min(T, (int)ceil((double)p.top_frac * (double)T));
    for (int i = tid; i < ktop; i += kTopkThreads) kept[idx[i]] = 1;
    for (int c = tid; c < T; c += kTopkThreads)
        if (c == 0 || c >= T - p.keep_last) kept[c] = 1;
    __syncthreads();
    // output positions: block 0 first, then the other kept blocks in the requested
    // order, by a block-wide exclusive scan over the candidates j: block T - 1 - j
    // (descending index) or the block of rank j (descending score)
    constexpr int PER = kMaxSelectBlocks / kTopkThreads;
    auto cand = [&](int j) -> int { return p.by_score ? (j < T ? idx[j] : 0) : T - 1 - j; };
    int f[PER], run = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int c = cand(tid * PER + k);
        f[k] = (c >= 1 && c < T && kept[c]) ? 1 : 0;
        run += f[k];
    }
    const int lane = tid & 31, wid = tid >> 5;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int ws = lane < kTopkThreads / 32 ? s_wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += v;
        }
        if (lane < kTopkThreads / 32) s_wsum[lane] = ws;  // inclusive per warp
    }
    __syncthreads();
    int pos = 1 + (incl - run) + (wid > 0 ? s_wsum[wid - 1] : 0);  // after block 0
    const int total = 1 + s_wsum[kTopkThreads / 32 - 1];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int c = cand(tid * PER + k);
        if (f[k]) {
            if (pos < p.max_visit) out[pos] = c;
            ++pos;
        }
    }
    if (tid == 0 && T > 0) out[0] = 0;
    for (int i = (T > 0 ? total : 0) + tid; i < p.max_visit; i += kTopkThreads) out[i] = -1;
}

size_t select_workspace_bytes(const art_shape& s) {
    const long long maxT = ((long long)s.max_pages_per_seq * s.page_size + kBK - 1) / kBK;
    return sizeof(WsHeader) + (size_t)s.batch * s.num_kv_heads * (size_t)maxT * sizeof(float);
}

}  // namespace art

using namespace art;

extern "C" {

size_t art_select_workspace_bytes(const art_shape* shape) {
    if (!shape || shape->batch < 1 || shape->num_kv_heads < 1 || shape->max_pages_per_seq < 1 || shape->page_size < 1)
        return 0;
    return select_workspace_bytes(*shape);
}

int art_select_blocks(const void* q, const void* k_cache, const int32_t* block_table, const int32_t* seq_lens,
                      float top_frac, int32_t keep_last, int32_t order, int32_t* visit_order, const art_shape* shape,
                      void* workspace, size_t workspace_bytes, void* stream) {
    if (!shape || !q || !k_cache || !block_table || !seq_lens || !visit_order || !workspace) return ART_ERR_INVALID_ARG;
    const art_shape& s = *shape;
    if (s.batch < 1 || s.num_q_heads < 1 || s.num_kv_heads < 1 || s.num_q_heads % s.num_kv_heads != 0 ||
        s.page_size < 1 || s.max_pages_per_seq < 1 || s.max_visit < 1 || s.num_pages_total < 1)
        return ART_ERR_INVALID_ARG;
    if (s.dtype != ART_DTYPE_BF16 && s.dtype != ART_DTYPE_F32) return ART_ERR_INVALID_ARG;
    if (s.head_dim != 64 && s.head_dim != 128) return ART_ERR_UNSUPPORTED;
    if (s.block_size != kBK) return ART_ERR_UNSUPPORTED;
    if (!(top_frac >= 0.f && top_frac <= 1.f) || keep_last < 0 || (order != 0 && order != 1))
        return ART_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_cache) & 15u) || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return ART_ERR_INVALID_ARG;
    const long long maxT = ((long long)s.max_pages_per_seq * s.page_size + kBK - 1) / kBK;
    if (maxT > kMaxSelectBlocks) return ART_ERR_UNSUPPORTED;
    if ((long long)s.batch * s.num_kv_heads > (1LL << 24)) return ART_ERR_UNSUPPORTED;
    // the longest possible list must fit a visit_order row
    const long long need = (long long)ceil((double)top_frac * (double)maxT) + 1 + keep_last;
    if (s.max_visit < (need < maxT ? need : maxT)) return ART_ERR_INVALID_ARG;
    if (workspace_bytes < select_workspace_bytes(s)) return ART_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = static_cast<WsHeader*>(workspace);
    cudaError_t e = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st);
    if (e != cudaSuccess) return cuda_fail(e);
    SelectParams p;
    p.q = q;
    p.k = k_cache;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.scores = reinterpret_cast<float*>(hdr + 1);
    p.visit = visit_order;
    p.hdr = hdr;
    p.B = s.batch;
    p.Hq = s.num_q_heads;
    p.Hkv = s.num_kv_heads;
    p.Ps = s.page_size;
    p.max_pages = s.max_pages_per_seq;
    p.max_visit = s.max_visit;
    p.num_pages = s.num_pages_total;
    p.maxT = (int)maxT;
    p.keep_last = keep_last;
    p.by_score = order;
    p.top_frac = top_frac;
    const int items = s.batch * s.num_kv_heads;
    const dim3 grid((unsigned)((maxT + kScoreBlocksPerCta - 1) / kScoreBlocksPerCta), (unsigned)items);
    const bool bf = s.dtype == ART_DTYPE_BF16;
    if (bf && s.head_dim == 128) art_score_kernel<true, 128><<<grid, kScoreThreads, 0, st>>>(p);
    else if (bf) art_score_kernel<true, 64><<<grid, kScoreThreads, 0, st>>>(p);
    else if (s.head_dim == 128) art_score_kernel<false, 128><<<grid, kScoreThreads, 0, st>>>(p);
    else art_score_kernel<false, 64><<<grid, kScoreThreads, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    const size_t smem = (size_t)kMaxSelectBlocks * (2 * sizeof(float) + sizeof(int));
    if ((e = cudaFuncSetAttribute(art_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return cuda_fail(e);
    art_topk_kernel<<<items, kTopkThreads, smem, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
    return ART_OK;
}

}  // extern "C"
