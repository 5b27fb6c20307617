/*
 * art.h -- C ABI of the ART decode-attention library (libart).
 *
 * ART (Attention Run-time Termination; Qiu, Li, Kalnis, arXiv 2606.00024) is
 * block-wise decode attention over a paged KV cache that stops reading a
 * (sequence, KV head)'s remaining KV blocks once a probe of its partial output
 * has been stable for `patience` consecutive blocks.
 *
 *   Attention:            O = softmax(q K^T / sqrt(d)) V
 *                         (ART paper sec. 3.1, Eq. (1))
 *   Partial outputs:      O^(i) = output after the first i listed KV blocks
 *                         (sec. 3.1; converges to the full output)
 *   Probe:                x^(i) = O^(i) at a fixed set of head-dim indices,
 *                         concatenated over the G query heads of the KV head
 *                         (sec. 3.2 probe vector)
 *   Stability test:       d_mag = | ||x^(i)|| - ||x^(i-1)|| | / ||x^(i-1)||
 *                         d_dir = 1 - cos(x^(i), x^(i-1))
 *                         stable iff d_mag < eps_mag and d_dir < eps_dir
 *                         (gist.science explainer of the paper, sec. 2.2)
 *   Patience:             stop after `patience` consecutive stable blocks
 *                         (explainer sec. 2.3)
 *   Block 0:              never stop before logical block 0, when it is listed,
 *                         has been processed (explainer sec. 2.4)
 *   Visit order:          a free input, e.g. the attention sink first and then
 *                         most recent first (explainer sec. 2.4)
 *
 * Conventions for every entry point
 *   - Array pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t passed
 *     as void*, 0 = legacy default stream); nothing synchronizes the host.
 *   - The return value is ART_OK or a negative ART_ERR_* code from host-side
 *     argument checks or the launch. Problems that only show in device data
 *     (a visit entry or page id out of range, a duplicate visit entry, a
 *     probe index out of range or repeated) never fault: the item gets
 *     blocks_used = -1 and a zero output, and a bit is set in the device
 *     status word (art_read_device_status).
 *
 * Layouts (row-major, element type bf16 or fp32 as given by shape->dtype)
 *   q            [batch][num_q_heads][head_dim]
 *   k_cache      [num_pages_total][num_kv_heads][page_size][head_dim]
 *   v_cache      same as k_cache
 *   block_table  int32 [batch][max_pages_per_seq]: physical page of each
 *                logical page; entries past ceil(seq_len / page_size) are
 *                never read
 *   seq_lens     int32 [batch], 0 <= seq_len <= max_pages_per_seq * page_size
 *   visit_order  int32 [batch][num_kv_heads][max_visit]: logical ART-block ids
 *                (block c holds tokens [c*block_size, (c+1)*block_size)), in
 *                visit order, ended by the first -1 or by max_visit entries;
 *                entries must be distinct and lie in [0, ceil(seq_len/block_size)).
 *                NULL means the natural order 0, 1, ..., ceil(seq_len/block_size)-1.
 *   probe_idx    int32 [num_probe]: distinct head-dim indices in [0, head_dim)
 *   out          [batch][num_q_heads][head_dim], same dtype as q
 *   blocks_used  int32 [batch][num_kv_heads]
 *   Query head h is served by KV head h / (num_q_heads / num_kv_heads).
 *
 * Alignment: q, k_cache, v_cache, out and workspace must be 16-byte aligned.
 *
 * Supported: dtype bf16 or fp32; head_dim 64 or 128; group size
 * G = num_q_heads / num_kv_heads in {1, 2, 4, 7, 8}; block_size 64;
 * page_size a power of two from 8 to 4096; num_probe 1..32, or for bf16 up to
 * head_dim (a probe over every head dim: the ablation of the gist.science
 * explainer sec. 4 and the ART paper sec. 3.2, whose probe is a subset of the
 * head dims; such calls always run one CTA per item).
 */
#ifndef ART_H_
#define ART_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct art_shape {
    int32_t batch;             /* B                                           */
    int32_t num_q_heads;       /* Hq                                          */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0                          */
    int32_t head_dim;          /* d                                           */
    int32_t page_size;         /* tokens per KV-cache page                    */
    int32_t block_size;        /* tokens per ART block (the unit of the test) */
    int32_t max_pages_per_seq; /* columns of block_table                      */
    int32_t max_visit;         /* last dimension of visit_order               */
    int32_t num_probe;         /* m, entries of probe_idx                     */
    int32_t num_pages_total;   /* pages in k_cache / v_cache                  */
    int32_t dtype;             /* ART_DTYPE_BF16 or ART_DTYPE_F32             */
} art_shape;

enum { ART_DTYPE_BF16 = 0, ART_DTYPE_F32 = 1 };

enum {
    ART_OK = 0,
    ART_ERR_INVALID_ARG = -1, /* null pointer, bad size, misalignment, bad eps/patience */
    ART_ERR_UNSUPPORTED = -2, /* a size outside the supported set above              */
    ART_ERR_WORKSPACE = -3,   /* workspace smaller than art_workspace_bytes()        */
    ART_ERR_LAUNCH = -4,      /* a CUDA call failed (see art_last_cuda_error)        */
};

/* Bits of the device status word. */
enum {
    ART_STATUS_BAD_VISIT = 1,   /* a visit entry outside [0, ceil(seq_len/block_size)) */
    ART_STATUS_DUP_VISIT = 2,   /* a block listed twice for one item                  */
    ART_STATUS_BAD_PAGE = 4,    /* a block_table entry of a listed block outside the pool */
    ART_STATUS_BAD_SEQLEN = 8,  /* seq_len < 0 or beyond the block table             */
    ART_STATUS_BAD_PROBE = 16,  /* probe index out of range or repeated              */
    ART_STATUS_TIMEOUT = 32,    /* a bounded wait inside the kernel gave up          */
    ART_STATUS_INTERNAL = 64,   /* an internal consistency check failed (the access was skipped) */
};

/* Bytes of device workspace art_decode / dense_decode need for `shape`.
 * Returns 0 if shape is NULL. For bf16 this includes the area of the unit path
 * (art_decode_path) when that area stays within 4 GiB; it grows with
 * batch * num_kv_heads and with max_pages_per_seq * page_size (the longest
 * possible list). A smaller workspace (at least the one-CTA path's part) keeps
 * every call on the one-CTA path. */
size_t art_workspace_bytes(const art_shape* shape);

/*
 * Which kernel path art_decode takes for these arguments on the current device
 * (an addition of this library; the ART paper describes one CTA per sequence):
 *   0  one CTA per item (b, g) at a time: a persistent kernel whose CTAs claim
 *      whole items, longest lists first (bf16: one CTA per SM whose three
 *      consumer groups, four when there are no more items than SMs, take
 *      alternate blocks of the item);
 *   1  the unit path: each item's list is cut into units of 8 to 16 blocks
 *      (chosen per call so that the units fill whole waves of CTAs) that any
 *      CTA may take, so one item is spread over many SMs; the stop is
 *      found from per-unit statistics joined by a look-back, the blocks of
 *      the stopping unit up to the stop are recomputed, and a second kernel
 *      merges the units' partial outputs. Blocks of units claimed before the
 *      stop was known are read and discarded.
 * The unit path is taken for bf16 when batch * num_kv_heads is below the
 * number of SMs / 2, patience <= 16, num_probe <= 32 and workspace_bytes covers
 * its area; the environment variable ART_UNITS=0 or 1 forces the choice where
 * the path is offered (any batch size). A shape that fails the argument checks
 * returns 0.
 */
int art_decode_path(const art_shape* shape, int32_t patience, size_t workspace_bytes);

/* The kernel path dense_decode takes (0 or 1 as above). The full scan has no
 * stop to find: it takes the unit path (all units, no statistics, no recompute)
 * where that path is offered (bf16 and a workspace that covers its area) and
 * batch * num_kv_heads is below the number of SMs; with more items one CTA per
 * SM streams as fast or faster. ART_UNITS=0 or 1 forces the choice as above. An
 * addition of this library. */
int dense_decode_path(const art_shape* shape, size_t workspace_bytes);

/*
 * ART decode attention (the method of the ART paper, sec. 3; the rule of the
 * explainer, sec. 2.2-2.4). For every item (b, g) it visits the listed KV
 * blocks in order, accumulates softmax attention for the G query heads of KV
 * head g, and after block i evaluates the stability test on the probe of
 * O^(i). It stops at the first i where `patience` consecutive tests passed
 * and logical block 0 (if listed) has been processed; blocks after i are
 * neither computed nor copied further (at most the blocks already in flight
 * are read; on the unit path, art_decode_path, the units already claimed).
 *   eps_mag, eps_dir: thresholds tau and phi, >= 0 (+inf disables a test,
 *                     0 makes the test never pass)
 *   patience:         p >= 1
 *   out:              O^(blocks_used) per query head
 *   blocks_used:      i per item (0 for an empty list, -1 for a bad item)
 *   workspace:        device scratch of art_workspace_bytes(shape) bytes; the
 *                     call zeroes what it needs on `stream`. Concurrent calls
 *                     must use separate workspaces.
 */
int art_decode(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_table, const int32_t* seq_lens,
               const int32_t* visit_order, float eps_mag, float eps_dir,
               int32_t patience, const int32_t* probe_idx, void* out,
               int32_t* blocks_used, const art_shape* shape, void* workspace,
               size_t workspace_bytes, void* stream);

/* Options of art_decode_ex (an addition of this library for ablations). */
typedef struct art_options {
    int32_t probe_heads; /* 0: the probe concatenates all G query heads of the
                            group (art_decode); 1..G: only heads 0..probe_heads-1
                            (probe_heads = 1 is closest to the ART paper's probe,
                            a fragment of one head's output, sec. 3.2) */
    int32_t reserved[7]; /* must be zero */
} art_options;

/* art_decode with options (NULL: the defaults, i.e. art_decode). A
 * probe_heads outside 0..G or a non-zero reserved field: ART_ERR_INVALID_ARG. */
int art_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_table, const int32_t* seq_lens,
                  const int32_t* visit_order, float eps_mag, float eps_dir,
                  int32_t patience, const int32_t* probe_idx, void* out,
                  int32_t* blocks_used, const art_shape* shape, void* workspace,
                  size_t workspace_bytes, void* stream, const art_options* options);

/*
 * The full-scan twin: the same blocked attention over every listed block,
 * with no probe, no test and no termination. probe_idx and num_probe are not
 * used. Items with bad device data get a zero output and a status bit.
 */
int dense_decode(const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_table, const int32_t* seq_lens,
                 const int32_t* visit_order, void* out, const art_shape* shape,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * art_decode without a caller-provided workspace. (An addition of this
 * library; the ART paper has no counterpart.)
 *
 * Some callers cannot allocate device memory: for example a plug-in running
 * inside a host framework that owns every device allocation through its own
 * pool, or a decode loop whose latency budget rules out allocator calls. This
 * entry point takes the same arguments as art_decode except the workspace,
 * and keeps its scratch (the 64-byte header, per-item {n, flags} and the
 * claim order) in a device array compiled into the library: 196,864 bytes per
 * device that loads the library, held until the process exits. It calls no
 * device allocator.
 *   Limit: batch * num_kv_heads <= 16384; larger calls return
 *          ART_ERR_UNSUPPORTED without touching the device.
 *   Set-up: every call looks up the array's device address on the current
 *          device (cudaGetSymbolAddress, which allocates nothing), so a
 *          device reset cannot leave a stale address behind. The first call
 *          on a device may load the library's device code: make it before
 *          any stream capture.
 *   Sharing: every call on a device uses the same array. Each call clears
 *          what must start at zero on `stream`, but calls that overlap on the
 *          GPU (other streams, other threads) race on it and must be ordered
 *          by the caller. Its status word is read with art_read_static_status.
 */
int art_decode_static(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* seq_lens,
                      const int32_t* visit_order, float eps_mag, float eps_dir,
                      int32_t patience, const int32_t* probe_idx, void* out,
                      int32_t* blocks_used, const art_shape* shape, void* stream);

/* Copies the status word of art_decode_static's array on the current device
 * (the ART_STATUS_* bits of the last call there; a blocking copy: call it
 * after the stream has finished that call). An addition of this library; the
 * ART paper has no counterpart. Returns ART_OK, ART_ERR_INVALID_ARG for a
 * NULL `status`, or ART_ERR_LAUNCH. */
int art_read_static_status(int32_t* status);

/*
 * Key-based block selection: writes a visit list for art_decode (ART paper
 * sec. 4, ART composed with key-centric KV selection; the score is the pooled
 * block estimate of the FlexPrefill summary). For every item (b, g), with
 * T = ceil(seq_len / block_size):
 *   score_c = mean over the G query heads of g (q_h) . mean over the tokens
 *             t < seq_len of block c (k_t)                      (fp32)
 *   kept    = the ceil(top_frac * T) highest scores (equal scores: the lower
 *             block index first), block 0, and the last keep_last blocks
 *   visit_order[b][g][:] = 0, then the other kept blocks, then -1 up to
 *             max_visit; order 0: by descending index (most recent first),
 *             order 1: by descending score (importance first; equal scores:
 *             the lower block index first) -- the two visit orders the ART
 *             paper sec. 4 discusses.
 *   top_frac in [0, 1]; keep_last >= 0; block_size 64; head_dim 64 or 128;
 *   T <= 8192 (max_pages_per_seq * page_size <= 524288 tokens).
 *   shape->max_visit must hold the longest possible list,
 *   min(T_max, ceil(top_frac * T_max) + 1 + keep_last) with
 *   T_max = ceil(max_pages_per_seq * page_size / block_size), else
 *   ART_ERR_INVALID_ARG. num_probe and probe indices are not used.
 *   workspace:  device scratch of art_select_workspace_bytes(shape) bytes (a
 *               header with the status word, then the block scores); zeroed
 *               as needed on `stream`. A page id outside the pool or a bad
 *               seq_len gives the item an empty list and a status bit.
 * Asynchronous on `stream`, like art_decode.
 */
size_t art_select_workspace_bytes(const art_shape* shape);
int art_select_blocks(const void* q, const void* k_cache, const int32_t* block_table,
                      const int32_t* seq_lens, float top_frac, int32_t keep_last,
                      int32_t order, int32_t* visit_order, const art_shape* shape,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Copies the device status word out of `workspace` (a blocking copy; call it
 * after the stream has finished the call of interest). Returns ART_OK or
 * ART_ERR_INVALID_ARG / ART_ERR_LAUNCH. */
int art_read_device_status(const void* workspace, int32_t* status);

/* Static text for a return code. */
const char* art_status_string(int code);

/* Text of the last CUDA error seen by this library in the calling thread. */
const char* art_last_cuda_error(void);

/*
 * Measurement hook (an addition of this library; the ART paper has none).
 * `start` and `stop` are cudaEvent_t handles passed as void*, owned by the
 * caller. While set, every art_decode / dense_decode / art_decode_static call
 * made by the calling thread records `start` on its stream right before the
 * decode-kernel launch and `stop` right after it, so that cudaEventElapsedTime
 * gives the decode kernel alone (without the workspace memset and the plan
 * kernel). A call that fails its checks records neither. NULL, NULL clears.
 */
void art_set_timing_events(void* start, void* stop);

#ifdef __cplusplus
}
#endif

#endif /* ART_H_ */
