// art_kernel.cuh -- the persistent, warp-specialized ART decode-attention kernel.
//
// One CTA runs these roles over a ring of shared-memory slots, each slot
// holding one 64-token ART block of K rows, V rows and (with a consumer
// group's first block of an item) the item's G query vectors:
//
//   producer warp    claims work items (sequence b, KV head g) in the order the
//                    plan kernel wrote (longest visit list first) and resolves
//                    visit entry -> logical block -> physical pages through the
//                    block table. For each ring entry it waits for the slot and
//                    writes the slot's metadata; with copy warps it posts a copy
//                    job (the pages' rows in the tensor maps), otherwise it
//                    issues the copies itself (fp32: one bulk copy per page).
//                    It posts no more blocks of an item once the statistics
//                    warp has stopped it.
//   copy warps       (bf16, one CTA per SM) take alternate ring entries, arm the
//                    slot's mbarrier with the entry's bytes and issue its copies
//                    (one 3-D tensor copy per page of K and of V, and the
//                    queries). A tensor copy holds the issuing warp until the
//                    copy engine accepts it, so issuing apart from resolving
//                    lets the two overlap.
//   consumer warps   softmax attention of the block for the item's G query
//                    heads and the online-softmax fold into running
//                    accumulators (ART paper sec. 3.1: FlashAttention's
//                    streaming softmax, O^(t) after t blocks). Three forms:
//                    - fp32: 8 warps on CUDA cores (packed f32x2 FMA), each
//                      owning 8 of the block's rows;
//                    - bf16, groups of 4 warps with the head dims split: three
//                      groups by default, four when each CTA runs one item,
//                      or one for a probe over more than 32 columns per head;
//                    - bf16, one or two groups of 4 warps with the keys split
//                      (when forced with ART_GROUPS).
//                    Several groups of one CTA take alternate blocks of the
//                    same item and merge their accumulators at its end.
//   statistics warp  (ART only) forms, in visit order, the probe x^(i) of O^(i)
//                    from the blocks' partials and evaluates the stability
//                    test (magnitude and direction change both below their
//                    thresholds for `patience` consecutive blocks, never
//                    before block 0 has been processed) -- ART paper sec. 3.2,
//                    gist.science explainer sec. 2.2-2.4.
//
// A consumer group folds block i into its accumulators only when block i's
// decision has arrived, one block later (the fp32 warps with G > 4, short of
// registers, wait for each block's own decision); a block computed past a stop
// is discarded. Where no stop is possible at a block, the statistics warp sends
// "continue" before computing the block's statistics.
//
// The statistics avoid cancellation: the change of the probe over block i is
// formed directly, delta = b (P.V_probe - l_blk x^(i-1)) / L_i, the norm
// change as delta.(2x + delta) / (|x_i| + |x_{i-1}|), and 1 - cos as
// |x_i/|x_i| - x_{i-1}/|x_{i-1}||^2 / 2.
//
// Every mbarrier wait is bounded (Params::wait_ns, 1 s); on expiry the kernel
// sets ART_STATUS_TIMEOUT, the warps that issued copies wait for their own
// copies in flight, and the CTA returns.
#pragma once

#include <cstddef>
#include <cstdlib>
#include <cstring>

#include "art_common.cuh"

namespace art {

__host__ __device__ constexpr int pow2ceil(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}
__host__ __device__ constexpr int imax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

enum Decision : int { kContinue = 0, kStop = 1, kDiscard = 2 };

// kSplitDims: one group of four tensor-core warps with the head dims split (the unit
// kernel's consumers, and the variant for probes over more than kMaxProbe columns);
// otherwise three or four groups split the dims, one or two the keys.
// kMP: probe columns per query head at most (kMaxProbe, or D for a probe over every
// head dim).
template <bool kBF16, int D, int G, int kNG = 1, bool kSplitDims = false, int kMP = kMaxProbe>
struct Cfg {
    using E = Elem<kBF16>;
    static constexpr bool TC = kBF16;            // bf16: tensor-core consumers on swizzled tiles
    static constexpr int NG = TC ? kNG : 1;      // consumer groups (alternate ring entries of one item)
    static constexpr int GW = TC ? 4 : 8;        // warps per consumer group
    static constexpr int NWC = NG * GW;          // consumer warps
    // record buffers: a group publishes entry u after the decision on u - 2 NG, which the
    // statistics warp may send before it has read u - 2 NG's partials, so NB > 2 NG; a
    // multiple of NG keeps each buffer (and its decision word) with one group
    static constexpr int NB = TC ? 3 * NG : 2;
    // four tensor-core groups split the head dims between the warps of a group
    // (fewer registers per warp); one or two groups, and the fp32 warps, split the keys
    static constexpr bool DS = TC && (NG >= 3 || kSplitDims);
    // rows of block partials per record: with the dims split each probe column has
    // one writer; with the keys split, one row set per warp
    static constexpr int RGW = DS ? 1 : GW;
    static constexpr int DW = D / GW;            // tensor-core path: head dims per consumer warp
    static constexpr int MT = DW / 16;           // ... and its O^T m-tiles
    // tensor-core path with one CTA per SM (two or more groups): copy warps issue the
    // tensor copies of the entries the producer warp has resolved, alternate entries
    // each. A tensor copy holds the issuing warp for about as long as the copy engine
    // takes to accept it; apart, the warps' work overlaps. (Two CTAs per SM have two
    // producers already.)
    static constexpr bool COPYW = TC && NG >= 2;
    // copy warps: two with three groups (whose ring depth is even), else one
    static constexpr int NCW = COPYW ? (NG == 3 ? 2 : 1) : 0;
    static constexpr int THREADS = (NWC + 2 + NCW) * 32;
    static constexpr int GQ = G;                 // query heads per KV head
    static constexpr int ELT = E::kBytes;
    static constexpr int DD = D;
    static constexpr int ROWB = D * ELT;         // bytes of one K or V row
    static constexpr int CB = ROWB / 8 <= 32 ? 8 : 16;  // bytes of a row one lane reads
    static constexpr int EPC = CB / ELT;         // elements per chunk
    static constexpr int E2 = EPC / 2;           // packed pairs per chunk
    static constexpr int LPR = ROWB / CB;        // lanes covering one row
    static constexpr int RPW = 32 / LPR;         // rows per warp instruction
    static constexpr int RW = kBK / GW;          // rows per consumer warp per block
    static constexpr int NI = RW / RPW;          // warp instructions per block
    static constexpr int NV = NI * G;            // partial scores per lane
    static constexpr int NVP = pow2ceil(imax(NV, LPR));
    static constexpr int QB = (int)align_up((size_t)G * D * ELT, 16);
    static constexpr int KVB = kBK * ROWB;       // bytes of K (or V) of one block
    static constexpr int SLOT = (int)align_up((size_t)2 * KVB + QB, TC ? 1024 : 16);
    // probe partial rows: word s * GP + h holds probe rank s of head h (GP even, so a
    // lane's pair of adjacent heads is one 8-byte store); rows padded by 8 words so
    // that the high- and low-part rows of the split tile fall in other banks
    static constexpr int GP = (G + 1) & ~1;
    static constexpr int MP = kMP;
    static constexpr int PST = kMP * GP + 8;
    static constexpr int SPL = (kMP * GP + 31) / 32;  // probe slots per stat lane
    static_assert(32 % GP == 0, "a stat lane's slots share one head");
    // G <= 4: the P.V products put the bf16 high parts of P in columns 0-3 of the
    // 8-wide tile and the low parts in columns 4-7, one mma per m-tile
    static constexpr bool SPLITN = TC && G <= 4;
    static constexpr int PRW = TC ? (SPLITN ? 2 : 1) : RPW;  // probe partial rows per warp
    static constexpr int PART_F = NB * RGW * PRW * PST;
    static constexpr int XBW = SPLITN ? 2 : 4;   // words of a lane's P^T fragment
    // bytes of a group's exchange area (dims split); the item-end merge reuses it
    static constexpr int XGB = (2 * GW * 32 * XBW + 2 * 2 * 8 * GW) * 4;
    static_assert(!TC || NG < 3 || XGB >= (G * D + 2 * G) * 4, "merge area fits the exchange area");
    static constexpr int KS = D / 16;            // tensor-core k-steps (QK) and m-tiles (PV)
    static constexpr bool LAG = G <= 4;          // decision one block behind (register budget)
    static constexpr bool HINT = TC && NG >= 3;  // bounded waits with a long suspend-time hint
    static_assert(LPR >= 8 && LPR <= 32 && EPC >= 2 && EPC <= 8, "row must be 128..512 bytes");
    static_assert(RW % RPW == 0 && NI >= 1, "rows per warp");
    static_assert(TC || 32 % RW == 0, "softmax lane groups");
    static_assert(G >= 1 && G <= 8, "group size");
};

struct alignas(16) SlotMeta {  // read as three 16-byte words
    int item, pos, n, c, nvalid, kind, b, g, has0, pad0, pad1, pad2;
};

// What the copy warp loads into a ring entry (tensor-core path).
enum JobKind : int { kJobData = 0, kJobNone = 1, kJobEnd = 2 };
struct SlotJob {
    int kind;    // kJobData: npg pages of K and of V (and the queries when with_q); otherwise no data
    int npg;     // pages of the block, 1..8
    int with_q;  // the entry also carries the item's queries
    int b, g;    // sequence and KV head (the queries' address)
    int y[8];    // first cache row of each page in the tensor map: (page * Hkv + g) * Ps + first row
    int pad0, pad1, pad2;
};
static_assert(sizeof(SlotJob) == 64, "four 16-byte words");

constexpr int kMaxNB = 16;  // record buffers at most (4 per consumer group)

struct Ctrl {
    int dec[kMaxNB];
    int stop_item;
    int abort;
    unsigned long long wait_ns;  // limit of the bounded waits (Params::wait_ns)
    SlotMeta info[kMaxNB];  // item and position of each published record
};
static_assert(offsetof(Ctrl, wait_ns) % 8 == 0, "8-byte field");

struct Layout {
    size_t meta, job, bars, part, plb, pmb, wmax, scr, eacc, qt, xb, sh, ptab, ctrl, total;
};

template <class C>
__host__ __device__ inline Layout make_layout(int stages) {
    constexpr int G = C::GQ;
    Layout L;
    size_t o = (size_t)stages * C::SLOT;
    L.meta = o;
    o += (size_t)stages * sizeof(SlotMeta);
    o = align_up(o, 16);
    L.job = o;  // copy warps: [stages] jobs, then [stages] the last data entry each slot received
    o += C::COPYW ? (size_t)stages * (sizeof(SlotJob) + sizeof(int)) : 0;
    o = align_up(o, 16);
    L.bars = o;
    // full, empty, record-full, decision [NB], cbar, the stall barrier, then the jobs' barriers
    o += (size_t)(2 * stages + 2 * C::NB + 2 + (C::COPYW ? stages : 0)) * sizeof(uint64_t);
    o = align_up(o, 16);
    L.part = o;  // [NB][RGW][PRW][PST] probe partial rows
    o += (size_t)C::PART_F * sizeof(float);
    L.plb = o;  // [NB][RGW][G] block sums
    o += (size_t)C::NB * C::RGW * G * sizeof(float);
    L.pmb = o;  // [NB][RGW][G] block maxima
    o += (size_t)C::NB * C::RGW * G * sizeof(float);
    L.wmax = o;  // fp32 path: [2][NWC][8] per-warp maxima of the block being processed (by block parity)
    o += C::TC ? 0 : (size_t)2 * C::NWC * 8 * sizeof(float);
    L.scr = o;  // fp32 path: [NWC][G][RW] scores, then weights
    o += C::TC ? 0 : (size_t)C::NWC * G * C::RW * sizeof(float);
    o = align_up(o, 16);
    L.eacc = o;  // per consumer warp: [G][D] output sums, then [G] weight sums, then [G] maxima
                 // (dims split: per group, in the group's exchange area, which is idle then)
    o += C::DS ? 0 : (size_t)C::NWC * (G * C::DD + 2 * G) * sizeof(float);
    o = align_up(o, 1024);
    L.qt = o;  // tensor-core path, per group: the item's queries, 8 rows (heads past G zero), 128B-swizzled
    o += C::TC ? (size_t)C::NG * 8 * C::ROWB : 0;
    o = align_up(o, 16);
    L.xb = o;  // dims split, per group: [2 block parities][GW warps][32 lanes] P^T fragments,
               // then [2][8 heads][GW] block max exponents, then [2][8][GW] weight sums
    o += C::DS ? (size_t)C::NG * C::XGB : 0;
    if (C::DS) L.eacc = L.xb;
    o = align_up(o, 16);
    L.sh = o;  // [3][G] statistics warp scratch
    o += (size_t)3 * G * sizeof(float);
    o = align_up(o, 16);
    L.ptab = o;  // CUDA-core path: mask and base per chunk; tensor-core path: rank per column
    o += (size_t)(2 * C::LPR + C::DD) * sizeof(int);
    o = align_up(o, 16);
    L.ctrl = o;
    o += sizeof(Ctrl);
    L.total = align_up(o, 128) + (C::TC ? 1024 : 0);  // room to align the ring to 1024 bytes
    return L;
}

// ---------------------------------------------------------------------------
// warp helpers
// ---------------------------------------------------------------------------
// Sums v[] over groups of LPR consecutive lanes. On return lane j of a group
// (j = lane % LPR) holds, in v[0 .. NVP/LPR), the group sums of the original
// entries j*NVP/LPR .. (j+1)*NVP/LPR - 1.
template <int NVP, int LPR>
__device__ __forceinline__ void transpose_reduce(float (&v)[NVP], int lane) {
#pragma unroll
    for (int lvl = 0; (LPR >> (lvl + 1)) >= 1; ++lvl) {
        const int s = LPR >> (lvl + 1);
        const int half = NVP >> (lvl + 1);
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
    return x;
}

// Waits for the phase with `parity` of `bar` to complete, warp-uniformly.
// kHint: the threads sleep in mbarrier.try_wait with a long suspend-time hint
// (woken by the phase completing); otherwise they wait in plain try_wait (a
// potentially blocking test that returns at the phase's completion or after the
// hardware's own short time limit). Measured: the hint is 0.5 % faster with one
// CTA per SM running three or four consumer groups, plain try_wait 2-3 % faster
// with two CTAs per SM. Returns false (and sets ART_STATUS_TIMEOUT) when the wait
// exceeds the CTA's limit (Ctrl::wait_ns). Only a warp's own wait ends it: the warps of a consumer
// group always wait on the same barrier phases, so they give up together and
// none is left behind in a named barrier.
template <bool kHint = false>
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, Ctrl* ctrl, WsHeader* hdr,
                                             int where = 0) {
    constexpr uint32_t kSleepNs = 200000;  // upper bound of one sleep; the limit is checked between sleeps
    auto try_once = [&]() -> bool {
        return kHint ? mbar_try_wait_sleep(bar, parity, kSleepNs) : mbar_try_wait(bar, parity);
    };
    // a phase that has completed already costs one test
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    if (__all_sync(0xffffffffu, try_once())) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, try_once())) return true;
        int late = (threadIdx.x & 31) == 0 && global_ns() - t0 > ctrl->wait_ns;
        if (__any_sync(0xffffffffu, late)) {
            if ((threadIdx.x & 31) == 0) {
                st_volatile_shared(&ctrl->abort, 1);
                atomicOr(&hdr->status, ART_STATUS_TIMEOUT);
                if (where) record_check(hdr, where, (int)parity, (int)(threadIdx.x >> 5), 0);
            }
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
// Tensor-core path: the copies of one block (npg pages of K, then of V) and, with
// with_q, of the item's queries into the slot at dst, completing on bar (armed by the
// caller). Each page's rows land as [column half][rows] (128-byte rows, 128B-swizzled),
// pages one after another: one 3-D copy per page, or one 2-D copy per column half.
// yof(k) is page k's first row in the tensor maps.
template <class C, class YF>
__device__ __forceinline__ void issue_block_tc(const Params& p, unsigned char* dst, int npg, bool with_q, int b, int g,
                                               uint64_t* bar, const CUtensorMap* tk, const CUtensorMap* tv, YF yof) {
    constexpr int NH = C::ROWB / 128;  // 128-byte column halves of a row
    const int lane = threadIdx.x & 31;
    const int page_rows = p.Ps <= kBK ? p.Ps : kBK;
    const int nop = p.tma3d ? npg : npg * NH;  // copies of K (and of V)
    const int nbox = 2 * nop;
    for (int t = lane; t < nbox + (with_q ? 1 : 0); t += 32) {
        if (t < nbox) {
            const int kv = t / nop;
            const int rem = t - kv * nop;
            const int k = p.tma3d ? rem : rem / NH, hf = p.tma3d ? 0 : rem - (rem / NH) * NH;
            const int y = yof(k);
            unsigned char* d = dst + kv * C::KVB + (k * NH + hf) * page_rows * 128;
            if (p.tma3d)
                tma_load_3d(d, kv ? tv : tk, 0, y, 0, bar);
            else
                tma_load_2d(d, kv ? tv : tk, hf * 64, y, bar);
        } else {
            const char* src = static_cast<const char*>(p.q) + ((size_t)b * p.Hq + (size_t)g * C::GQ) * C::ROWB;
            bulk_g2s(dst + 2 * C::KVB, src, (uint32_t)(C::GQ * C::ROWB), bar);
        }
    }
}

template <class C, bool kART>
__device__ void producer_warp(const Params& p, unsigned char* ring, SlotMeta* meta, SlotJob* job, uint64_t* full,
                              uint64_t* empty, uint64_t* jobb, Ctrl* ctrl, const CUtensorMap* tk,
                              const CUtensorMap* tv) {
    constexpr int G = C::GQ;
    const int lane = threadIdx.x & 31;
    int slot = 0;
    uint32_t round = 0;
    bool have_slot = false;
    unsigned long long issued = 0;
    bool ok = true;

    auto acquire = [&]() -> bool {
        if (have_slot) return true;
        if (!wait_bounded<C::HINT>(&empty[slot], (round & 1u) ^ 1u, ctrl, p.hdr, 131)) return false;
        have_slot = true;
        return true;
    };
    auto advance = [&]() {
        have_slot = false;
        ++issued;
        if (++slot == p.stages) {
            slot = 0;
            ++round;
        }
    };
    // an entry without data; every consumer group gets one (kind, item) entry
    auto emit1 = [&](int kind, int item, int b, int g, int pos, int n) -> bool {
        if (!acquire()) return false;
        if (lane == 0) {
            SlotMeta& mt = meta[slot];
            mt.item = item; mt.pos = pos; mt.n = n; mt.c = -1; mt.nvalid = 0; mt.kind = kind;
            mt.b = b; mt.g = g; mt.has0 = 0;
            if constexpr (C::COPYW) {
                job[slot].kind = kind == kSlotEnd ? kJobEnd : kJobNone;
                job[slot].npg = pos;  // an end entry: its index among the NG end entries
                mbar_arrive(&jobb[slot]);
            } else {
                mbar_arrive(&full[slot]);
            }
        }
        __syncwarp();
        advance();
        return true;
    };
    auto emit = [&](int kind, int item, int b, int g) -> bool {
        for (int k = 0; k < C::NG; ++k)
            if (!emit1(kind, item, b, g, k, 0)) return false;
        return true;
    };

    for (;;) {
        int idx = 0;
        if (lane == 0) idx = (int)atomicAdd(&p.hdr->claim, 1u);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx >= p.num_items) {
            ok = emit(kSlotEnd, -1, 0, 0);
            break;
        }
        const int item = __ldg(&p.order[idx]);
        if (item < 0 || item >= p.num_items) {
            if (lane == 0) record_check(p.hdr, 1, idx, item, 0);
            ok = emit(kSlotEnd, -1, 0, 0);
            break;
        }
        const ItemInfo inf = p.info[item];
        const int b = item / p.Hkv, g = item - (item / p.Hkv) * p.Hkv;
        if (inf.flags & kItemBad) {
            if (!(ok = emit(kSlotFail, item, b, g))) break;
            continue;
        }
        if (inf.n <= 0) {
            if (!(ok = emit(kSlotEmpty, item, b, g))) break;
            continue;
        }
        const int n = inf.n;
        const int seq_len = __ldg(&p.seq_lens[b]);
        const int32_t* trow = p.block_table + (size_t)b * p.max_pages;
        const int32_t* vrow = p.visit ? p.visit + (size_t)item * p.max_visit : nullptr;
        const char* kbase = static_cast<const char*>(p.k);
        const char* vbase = static_cast<const char*>(p.v);
        bool item_done = false;
        int nis = 0;  // block entries issued for this item
        for (int base = 0; base < n && !item_done; base += 32) {
            // each lane resolves one listed position
            const int pos = base + lane;
            int c = 0, nvalid = 0, npv = 0, bad = 0, r0 = 0;
            int pg[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) pg[k] = 0;
            if (pos < n) {
                c = vrow ? __ldg(&vrow[pos]) : pos;
                const int t0 = c * kBK;
                if (c < 0 || t0 >= seq_len) {
                    bad = 1;
                } else {
                    nvalid = min(kBK, seq_len - t0);
                    if (p.Ps <= kBK) {
                        npv = (nvalid + p.Ps - 1) / p.Ps;
                        const int first = t0 / p.Ps;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (k < npv) pg[k] = __ldg(&trow[first + k]);
                    } else {
                        npv = 1;
                        pg[0] = __ldg(&trow[t0 / p.Ps]);
                        r0 = t0 % p.Ps;
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (k < npv && (pg[k] < 0 || pg[k] >= p.num_pages)) bad = 1;
                }
            }
            const int cnt = min(32, n - base);
            for (int j = 0; j < cnt; ++j) {
                if (kART && ld_volatile_shared(&ctrl->stop_item) == item) { item_done = true; break; }
                if (!acquire()) { ok = false; break; }
                if (kART && ld_volatile_shared(&ctrl->stop_item) == item) { item_done = true; break; }
                const int badj = __shfl_sync(0xffffffffu, bad, j);
                if (badj) {
                    if (lane == 0) atomicOr(&p.hdr->status, ART_STATUS_BAD_PAGE);
                    if (!(ok = emit(kSlotFail, item, b, g))) break;
                    nis = C::NG;  // every group got an entry of the item
                    item_done = true;
                    break;
                }
                const int posj = base + j;
                const bool with_q = posj < C::NG;  // each consumer group's first entry of the item
                if constexpr (C::COPYW) {
                    // the lane that resolved the position describes the entry; the copy warp
                    // loads it and completes the slot's barrier
                    if (lane == j) {
                        SlotMeta& mt = meta[slot];
                        mt.item = item; mt.pos = posj; mt.n = n; mt.c = c; mt.nvalid = nvalid; mt.kind = kSlotBlock;
                        mt.b = b; mt.g = g; mt.has0 = inf.flags & kItemHas0;
                        SlotJob& jb = job[slot];
                        jb.kind = kJobData; jb.npg = npv; jb.with_q = with_q ? 1 : 0; jb.b = b; jb.g = g;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (k < npv) jb.y[k] = (pg[k] * p.Hkv + g) * p.Ps + r0;
                        mbar_arrive(&jobb[slot]);
                    }
                } else {
                    const int cj = __shfl_sync(0xffffffffu, c, j);
                    const int nvj = __shfl_sync(0xffffffffu, nvalid, j);
                    const int npj = __shfl_sync(0xffffffffu, npv, j);
                    const int r0j = __shfl_sync(0xffffffffu, r0, j);
                    int pgj[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) pgj[k] = __shfl_sync(0xffffffffu, pg[k], j);
                    const uint32_t page_bytes = (uint32_t)((p.Ps <= kBK ? p.Ps : kBK) * C::ROWB);
                    const uint32_t bytes = 2u * npj * page_bytes + (with_q ? (uint32_t)(G * C::ROWB) : 0u);
                    unsigned char* dst = ring + (size_t)slot * C::SLOT;
                    if (lane == 0) {
                        SlotMeta& mt = meta[slot];
                        mt.item = item; mt.pos = posj; mt.n = n; mt.c = cj; mt.nvalid = nvj; mt.kind = kSlotBlock;
                        mt.b = b; mt.g = g; mt.has0 = inf.flags & kItemHas0;
                        mbar_arrive_expect_tx(&full[slot], bytes);
                    }
                    __syncwarp();
                    if constexpr (C::TC) {
                        issue_block_tc<C>(p, dst, npj, with_q, b, g, &full[slot], tk, tv, [&](int k) {
                            int pk = 0;
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                if (u == k) pk = pgj[u];
                            return (pk * p.Hkv + g) * p.Ps + r0j;
                        });
                    } else {
                        // one bulk copy per page of K and of V, and one of the queries
                        const int ncopy = 2 * npj + (with_q ? 1 : 0);
                        if (lane < ncopy) {
                            if (lane < 2 * npj) {
                                const int k = lane < npj ? lane : lane - npj;
                                int pk = 0;
#pragma unroll
                                for (int t = 0; t < 8; ++t)
                                    if (t == k) pk = pgj[t];
                                const size_t row0 = ((size_t)pk * p.Hkv + g) * p.Ps + r0j;
                                const char* src = (lane < npj ? kbase : vbase) + row0 * C::ROWB;
                                unsigned char* d = dst + (lane < npj ? 0 : C::KVB) + (size_t)k * page_bytes;
                                bulk_g2s(d, src, page_bytes, &full[slot]);
                            } else {
                                const char* src =
                                    static_cast<const char*>(p.q) + ((size_t)b * p.Hq + (size_t)g * G) * C::ROWB;
                                bulk_g2s(dst + 2 * C::KVB, src, (uint32_t)(G * C::ROWB), &full[slot]);
                            }
                        }
                    }
                }
                __syncwarp();
                advance();
                ++nis;
            }
            if (!ok) break;
        }
        if (!ok) break;
        // every consumer group takes part in the item (its end is merged jointly):
        // pads for the groups that got no block of it (short lists, early stops)
        for (int k = nis; k < C::NG && ok; ++k) ok = emit1(kSlotPad, item, b, g, k, max(n, k + 1));
        if (!ok) break;
    }

    if (!ok && !C::COPYW) {
        // aborting: wait (bounded) for this CTA's own copies still in flight (the copy
        // warp waits for those it issued)
        const unsigned long long lim = issued < (unsigned long long)p.stages ? issued : p.stages;
        int s = slot;
        uint32_t r = round;
        for (unsigned long long k = 0; k < lim; ++k) {
            if (--s < 0) { s = p.stages - 1; --r; }
            const unsigned long long t0 = global_ns();
            while (!__all_sync(0xffffffffu, mbar_try_wait(&full[s], r & 1u)) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// ---------------------------------------------------------------------------
// copy warp (tensor-core path)
// ---------------------------------------------------------------------------
// Copy warp cw of NCW takes the ring entries u = cw, cw + NCW, ... in order: for each
// job the producer posted, it arms the slot's full barrier with the entry's bytes and
// issues the tensor copies of its pages (K, then V) and of the queries, or completes
// the barrier at once for an entry without data. The ring depth is a multiple of NCW,
// so a slot's entries u, u + stages, ... all belong to one copy warp: the job barrier
// phase a warp waits for is neither older than its previous entry in the slot (which
// it has taken) nor newer (a slot is posted again only once consumed, which needs
// this warp's copies). It leaves after its last entry among the consumer groups' NG
// end entries (NG >= NCW, so every copy warp takes one of them). last[s] holds the
// last data entry slot s received; on an abort each copy warp waits for the copies of
// the slots whose last entry is its own (a later entry in a slot means the earlier
// one was consumed).
template <class C>
__device__ void copy_warp(const Params& p, unsigned char* ring, const SlotJob* job, int* last, uint64_t* full,
                          uint64_t* jobb, Ctrl* ctrl, const CUtensorMap* tk, const CUtensorMap* tv, int cw) {
    constexpr int G = C::GQ, NCW = C::NCW;
    static_assert(C::NG >= NCW, "every copy warp takes an end entry");
    const int lane = threadIdx.x & 31;
    const int page_rows = p.Ps <= kBK ? p.Ps : kBK;
    const uint32_t page_bytes = (uint32_t)(page_rows * C::ROWB);
    int end_last = -1;  // the last end entry, once one end entry has been seen
    bool ok = true;
    for (int u = cw;; u += NCW) {
        if (end_last >= 0 && u > end_last) break;
        const int slot = u % p.stages;
        if (!wait_bounded<C::HINT>(&jobb[slot], (uint32_t)(u / p.stages) & 1u, ctrl, p.hdr, 171)) {
            ok = false;
            break;
        }
        const SlotJob* jb = &job[slot];
        const int kind = jb->kind;
        if (kind == kJobData) {
            const int npg = jb->npg, with_q = jb->with_q;
            if (npg < 1 || npg > 8) {
                // not a job the producer writes: complete the slot without data
                if (lane == 0) record_check(p.hdr, 6, slot, npg, 0);
                mbar_arrive_if(lane == 0, &full[slot]);
            } else {
                const uint32_t bytes = 2u * npg * page_bytes + (with_q ? (uint32_t)(G * C::ROWB) : 0u);
                if (lane == 0) {
                    last[slot] = u;
                    mbar_arrive_expect_tx(&full[slot], bytes);
                }
                __syncwarp();
                issue_block_tc<C>(p, ring + (size_t)slot * C::SLOT, npg, with_q != 0, jb->b, jb->g, &full[slot], tk, tv,
                                  [&](int k) { return jb->y[k]; });
            }
        } else {
            if (kind == kJobEnd) {
                const int k = jb->npg;  // its index among the end entries
                end_last = u + (C::NG - 1 - (k >= 0 && k < C::NG ? k : C::NG - 1));
            }
            mbar_arrive_if(lane == 0, &full[slot]);
        }
        __syncwarp();
    }
    if (!ok) {
        // aborting: wait (bounded) for the copies this warp issued that may still be in flight
        for (int s = 0; s < p.stages; ++s) {
            const int v = ld_volatile_shared(&last[s]);
            if (v < 0 || v % NCW != cw) continue;
            const unsigned long long t0 = global_ns();
            while (!__all_sync(0xffffffffu, mbar_try_wait(&full[s], (uint32_t)(v / p.stages) & 1u)) &&
                   global_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// ---------------------------------------------------------------------------
// statistics warp (ART only)
// ---------------------------------------------------------------------------
template <class C>
__device__ void stat_warp(const Params& p, const float* part, const float* plb, const float* pmb, float* sh,
                          uint64_t* part_full, uint64_t* dec_bar, Ctrl* ctrl) {
    constexpr int G = C::GQ;
    constexpr int SPL = C::SPL;
    constexpr int NP = C::RGW * C::PRW;  // partial rows per record
    constexpr int NB = C::NB;
    (void)sh;
    const int lane = threadIdx.x & 31;
    const int m = p.m;
    // probe slot k = lane + 32 j is word k of a partial row: head k % GP, rank k / GP
    // (the statistics do not depend on the order of the probe coordinates); heads
    // from p.ph on are not part of the probe
    int hs[SPL];
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
        const int k = lane + 32 * j;
        hs[j] = (k % C::GP < p.ph && k / C::GP < m) ? k % C::GP : -1;
    }
    // every slot of this lane belongs to head lane % GP, whose running max and
    // weight sum the lane keeps
    const int hme = lane % C::GP < G ? lane % C::GP : 0;
    float M = -INFINITY, Lsum = 0.f;
    float X[SPL];
    float nprev = 0.f, rprev = 0.f;  // |x_{i-1}| and its reciprocal
    int counter = 0, seen0 = 0;
    int stopped_item = -1;
    auto reset = [&]() {
        M = -INFINITY;
        Lsum = 0.f;
#pragma unroll
        for (int j = 0; j < SPL; ++j) X[j] = 0.f;
        nprev = 0.f;
        rprev = 0.f;
        counter = 0;
        seen0 = 0;
    };
    auto send = [&](int vb, int dec) {
        __syncwarp();
        st_shared_if(lane == 0, &ctrl->dec[vb], dec);
        mbar_arrive_if(lane == 0, &dec_bar[vb]);
    };
    reset();
    for (int v = 0;; ++v) {
        const int vb = v % NB;
        if (!wait_bounded<C::HINT>(&part_full[vb], (uint32_t)(v / NB) & 1u, ctrl, p.hdr, 141)) return;
        // every load of the record at once, ahead of the branches on its kind (for a
        // record without a block the partial values are stale and go unused)
        constexpr int RGW = C::RGW;
        const SlotMeta rec = ctrl->info[vb];
        float rmb[RGW], rlb[RGW], rpp[SPL][NP];
#pragma unroll
        for (int w = 0; w < RGW; ++w) {
            rmb[w] = pmb[(vb * RGW + w) * G + hme];
            rlb[w] = plb[(vb * RGW + w) * G + hme];
        }
        {
            const float* pp = part + (size_t)vb * NP * C::PST;
#pragma unroll
            for (int j = 0; j < SPL; ++j)
#pragma unroll
                for (int r = 0; r < NP; ++r) rpp[j][r] = pp[r * C::PST + lane + 32 * j];
        }
        const SlotMeta* info = &rec;
        const int kind = info->kind, item = info->item;
        if (kind == kSlotEnd) return;
        if (item == stopped_item || kind == kSlotPad) {
            // computed ahead of the decision that stopped its item, a pad, or the
            // second group's copy of a failed / empty item
            send(vb, kDiscard);
            continue;
        }
        if (kind != kSlotBlock) {
            if (lane == 0) p.blocks_used[item] = kind == kSlotFail ? -1 : 0;
            reset();
            stopped_item = item;
            send(vb, kStop);
            continue;
        }
        const int pos = info->pos, n = info->n, c = info->c, has0 = info->has0;
        if (pos == 0) reset();
        if (c == 0) seen0 = 1;
        // the stop can only happen here if the patience count can reach p at this
        // block and block 0 (when listed) has been processed; otherwise the
        // consumers learn "continue" at once and the statistics follow
        const bool last = pos == n - 1;
        const bool may_stop = (counter + 1 >= p.patience) && (seen0 || !has0);
        bool sent = false;
        if (last || !may_stop) {
            send(vb, last ? kStop : kContinue);
            sent = true;
        }
        // block max and sum of this lane's head over the consumer warps (each warp
        // used its own max), new running max and sum, and the factor that moves
        // the probe: delta = cf * (PV_probe - l_blk * x)
        float sw[RGW];
        float mbk = -INFINITY;
#pragma unroll
        for (int w = 0; w < RGW; ++w) {
            sw[w] = rmb[w];
            mbk = fmaxf(mbk, sw[w]);
        }
        float lb = 0.f;
        if constexpr (RGW == 1) {
            sw[0] = 1.f;
            lb = rlb[0];
        } else {
#pragma unroll
            for (int w = 0; w < RGW; ++w) {
                sw[w] = sw[w] == -INFINITY ? 0.f : exp2f(sw[w] - mbk);  // a row set without valid keys adds nothing
                lb = fmaf(sw[w], rlb[w], lb);
            }
        }
        const float Mn = fmaxf(M, mbk);
        const float a = exp2f(M - Mn);
        const float bw = exp2f(mbk - Mn);
        const float Ln = fmaf(a, Lsum, bw * lb);
        const float cf = __fdividef(bw, Ln);  // Ln >= 1/2: the block's largest weight is at least 1/2
        M = Mn;
        Lsum = Ln;
        float s1 = 0.f, s2 = 0.f, s3 = 0.f;  // sum delta^2, sum delta . x_{i-1}, |x_i|^2
#pragma unroll
        for (int j = 0; j < SPL; ++j) {
            float pb = 0.f;
#pragma unroll
            for (int w = 0; w < RGW; ++w) {
                float pw = 0.f;
#pragma unroll
                for (int r = 0; r < C::PRW; ++r) pw += rpp[j][w * C::PRW + r];
                pb = RGW == 1 ? pw : fmaf(sw[w], pw, pb);
            }
            // slots past the probe (or past G) hold no data: no change
            const float d = hs[j] >= 0 ? cf * (pb - lb * X[j]) : 0.f;
            s1 = fmaf(d, d, s1);
            s2 = fmaf(d, X[j], s2);
            X[j] += d;
            s3 = fmaf(X[j], X[j], s3);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
            s3 += __shfl_xor_sync(0xffffffffu, s3, o);
        }
        // With S = |x_i| + |x_{i-1}| and T = |x_i|^2 - |x_{i-1}|^2 = 2 s2 + s1 (the difference
        // of squares formed directly):
        //   d_mag = |T| / (S |x_{i-1}|)
        //   d_dir = 1 - cos = |x_i/|x_i| - x_{i-1}/|x_{i-1}||^2 / 2
        //         = (s1 - 2 s2 (T/S) / |x_{i-1}| + (T/S)^2) / (2 s3), clamped at 0.
        // Both tests are taken multiplied through by their (positive) denominators, so
        // no division sits on the chain; 1/|x_{i-1}| comes from the previous block.
        const float ni = sqrtf(s3);
        const float S = ni + nprev, T = 2.f * s2 + s1;
        const bool mag_ok = fabsf(T) * rprev < p.eps_mag * S;
        const float Nd = fmaf(s1, S * S, fmaf(-2.f * s2 * T, S * rprev, T * T));
        const bool dir_ok = fmaxf(0.f, Nd) < 2.f * p.eps_dir * s3 * (S * S);
        const bool stable = pos >= 1 && nprev > 0.f && ni > 0.f && nprev < 1e30f && ni < 1e30f && mag_ok && dir_ok;
        nprev = ni;
        rprev = __fdividef(1.f, ni);  // a few ulp; the next block's tests only
        counter = stable ? counter + 1 : 0;
        const bool stop = last || (may_stop && counter >= p.patience);
        if (stop) {
            stopped_item = item;
            if (lane == 0) {
                p.blocks_used[item] = pos + 1;
                st_volatile_shared(&ctrl->stop_item, item);
            }
        }
        if (!sent) send(vb, stop ? kStop : kContinue);
    }
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
template <class C, bool kART>
__device__ void consumer_warps(const Params& p, unsigned char* ring, const SlotMeta* meta, uint64_t* full,
                               uint64_t* empty, uint64_t* part_full, uint64_t* dec_bar, uint64_t* cbar,
                               const Layout& L, unsigned char* smem, const int* pmask, const int* pbase,
                               Ctrl* ctrl) {
    constexpr int G = C::GQ;
    constexpr int EPC = C::EPC, E2 = C::E2, LPR = C::LPR, RPW = C::RPW, RW = C::RW, NI = C::NI;
    constexpr int D = C::DD;
    constexpr int kNWC = C::NWC;
    constexpr bool LAG = kART && C::LAG;
    using E = typename C::E;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane / LPR, ch = lane % LPR;
    float* part = reinterpret_cast<float*>(smem + L.part);
    float* plb = reinterpret_cast<float*>(smem + L.plb);
    float* pmb = reinterpret_cast<float*>(smem + L.pmb);
    float* wmax = reinterpret_cast<float*>(smem + L.wmax);
    float* scr = reinterpret_cast<float*>(smem + L.scr) + (size_t)w * G * RW;  // [G][RW]
    float* eacc = reinterpret_cast<float*>(smem + L.eacc);                   // [NWC][G*D + G]
    const float qscale = 1.4426950408889634f / sqrtf((float)D);
    const uint32_t my_mask = (uint32_t)pmask[ch];
    const int my_base = pbase[ch];
    const int ctid = threadIdx.x;  // 0 .. kNWC*32-1

    uint64_t qs[G][E2];    // pre-scaled queries of this lane's chunk
    uint64_t acc[G][E2];   // running P.V of this lane's rows (scale m_run)
    uint64_t tN[G][E2];    // block just computed
    uint64_t tP[G][E2];    // block waiting for its decision (LAG)
    float mrun[G], lrun[G], mbN[G], lbN[G], mbP[G], lbP[G];
    SlotMeta mP;
    mP.item = -1; mP.b = 0; mP.g = 0;
    int vP = 0;
    bool pending = false;

    auto reset = [&]() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mrun[h] = -INFINITY;
            lrun[h] = 0.f;
#pragma unroll
            for (int e = 0; e < E2; ++e) acc[h][e] = 0ull;
        }
    };
    reset();
#pragma unroll
    for (int h = 0; h < G; ++h) {
        mbN[h] = mbP[h] = lbN[h] = lbP[h] = 0.f;
#pragma unroll
        for (int e = 0; e < E2; ++e) { qs[h][e] = 0ull; tN[h][e] = 0ull; tP[h][e] = 0ull; }
    }

    int slot = 0;
    uint32_t round = 0;
    int v = 0;          // records published to the statistics warp
    uint32_t cbph = 0;  // consumer-barrier phase
    int bpar = 0;       // parity of the blocks computed (selects the wmax buffer)
    int stopped_item = -1;

    auto cbar_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(cbar);
        const bool r = wait_bounded<C::HINT>(cbar, cbph, ctrl, p.hdr);
        cbph ^= 1u;
        return r;
    };
    auto release = [&]() {
        __syncwarp();
        mbar_arrive_if(lane == 0, &empty[slot]);
    };
    auto advance = [&]() {
        if (++slot == p.stages) { slot = 0; ++round; }
    };
    auto out_index = [&](int b, int g, int h, int col) -> size_t {
        return ((size_t)b * p.Hq + (size_t)g * G + h) * D + col;
    };
    auto publish = [&](const SlotMeta& mt) -> int {  // returns the record number
        const int vb = v & 1;
        if (w == 0 && lane == 0) ctrl->info[vb] = mt;
        __syncwarp();
        mbar_arrive_if(lane == 0, &part_full[vb]);
        return v++;
    };
    auto wait_dec = [&](int rec) -> int {
        if (!wait_bounded<C::HINT>(&dec_bar[rec & 1], (uint32_t)(rec >> 1) & 1u, ctrl, p.hdr)) return -1;
        return ctrl->dec[rec & 1];
    };
    auto fold = [&](const uint64_t (&t)[G][E2], const float* mb, const float* lb) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mn = fmaxf(mrun[h], mb[h]);
            const float a = exp2f(mrun[h] - mn);
            const float bb = exp2f(mb[h] - mn);
            const uint64_t a2 = pk2(a, a), b2 = pk2(bb, bb);
#pragma unroll
            for (int e = 0; e < E2; ++e) acc[h][e] = fma2(b2, t[h][e], mul2(a2, acc[h][e]));
            lrun[h] = a * lrun[h] + bb * lb[h];
            mrun[h] = mn;
        }
    };
    // all warps share the block maxima, so the running maxima agree across warps;
    // the warps' partial sums are added in a fixed order (reproducible results)
    auto epilogue = [&](int b, int g) -> bool {
        float fa[G][EPC];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < E2; ++e) up2(acc[h][e], fa[h][2 * e], fa[h][2 * e + 1]);
#pragma unroll
        for (int s = LPR; s < 32; s <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPC; ++e) fa[h][e] += __shfl_xor_sync(0xffffffffu, fa[h][e], s);
        float* mine = eacc + (size_t)w * (G * D + 2 * G);  // this warp's [G][D] sums, then [G] weights
        if (half == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPC; ++e) mine[h * D + ch * EPC + e] = fa[h][e];
        }
        if (lane < G) {
            float l = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h)
                if (h == lane) l = lrun[h];
            mine[G * D + lane] = l;
        }
        if (!cbar_sync()) return false;
        for (int idx = ctid; idx < G * D; idx += kNWC * 32) {
            const int h = idx / D, col = idx - (idx / D) * D;
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int ww = 0; ww < kNWC; ++ww) {
                num += eacc[(size_t)ww * (G * D + 2 * G) + idx];
                den += eacc[(size_t)ww * (G * D + 2 * G) + G * D + h];
            }
            E::store(p.out, out_index(b, g, h, col), num / den);
        }
        return cbar_sync();  // eacc is free again
    };
    auto write_zero = [&](int b, int g) {
        for (int idx = ctid; idx < G * D; idx += kNWC * 32)
            E::store(p.out, out_index(b, g, idx / D, idx % D), 0.f);
    };
    // resolves the pending block; returns false on abort
    auto resolve_pending = [&]() -> bool {
        const int d = wait_dec(vP);
        if (d < 0) return false;
        fold(tP, mbP, lbP);
        pending = false;
        if (d == kStop) {
            if (!epilogue(mP.b, mP.g)) return false;
            reset();
            stopped_item = mP.item;
        }
        return true;
    };

    for (;;) {
        if (!wait_bounded<C::HINT>(&full[slot], round & 1u, ctrl, p.hdr)) return;
        const SlotMeta mt = meta[slot];
        if (mt.kind == kSlotEnd) {
            if (LAG && pending && !resolve_pending()) return;
            if (kART) publish(mt);
            return;
        }
        if (mt.kind != kSlotBlock) {
            release();
            if (LAG && pending && !resolve_pending()) return;
            if (mt.item != stopped_item) {
                write_zero(mt.b, mt.g);
                if (kART && wait_dec(publish(mt)) < 0) return;
                reset();
                stopped_item = mt.item;
            }
            advance();
            continue;
        }
        if (mt.item == stopped_item) {  // fetched before the stop became visible to the producer
            release();
            advance();
            continue;
        }
        const unsigned char* sK = ring + (size_t)slot * C::SLOT;
        const unsigned char* sV = sK + C::KVB;
        if (mt.pos == 0) {
            const unsigned char* sQ = sK + 2 * C::KVB;
            const uint64_t sc2 = pk2(qscale, qscale);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                uint64_t q2[E2];
                E::template load_pairs<C::CB>(sQ + (size_t)h * C::ROWB + ch * C::CB, q2);
#pragma unroll
                for (int e = 0; e < E2; ++e) qs[h][e] = mul2(q2[e], sc2);
            }
        }
        const int nvalid = mt.nvalid;

        // ---- scores of this warp's rows: packed partial dots, transposed reduction
        float sv[C::NVP];
#pragma unroll
        for (int i = 0; i < C::NVP; ++i) sv[i] = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int r = w * RW + i * RPW + half;
            if (r < nvalid) {
                uint64_t k2[E2];
                E::template load_pairs<C::CB>(sK + (size_t)r * C::ROWB + ch * C::CB, k2);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    uint64_t d2 = 0ull;
#pragma unroll
                    for (int e = 0; e < E2; ++e) d2 = fma2(qs[h][e], k2[e], d2);
                    float lo, hi;
                    up2(d2, lo, hi);
                    sv[i * G + h] = lo + hi;
                }
            }
        }
        transpose_reduce<C::NVP, LPR>(sv, lane);
        constexpr int PER = C::NVP / LPR;
#pragma unroll
        for (int t = 0; t < PER; ++t) {
            const int idx = ch * PER + t;
            if (idx < C::NV) {
                const int i = idx / G, h = idx - (idx / G) * G;
                const int rl = i * RPW + half;
                scr[h * RW + rl] = (w * RW + rl < nvalid) ? sv[t] : -INFINITY;
            }
        }
        __syncwarp();

        // ---- block max per head: this warp's rows, then across warps
#pragma unroll
        for (int k = 0; k < (G * RW + 31) / 32; ++k) {
            const int idx = k * 32 + lane;
            const int h = idx / RW, rl = idx % RW;
            float mx = h < G ? scr[h * RW + rl] : -INFINITY;
#pragma unroll
            for (int o = RW / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (h < G && rl == 0) wmax[(bpar * kNWC + w) * 8 + h] = mx;
        }
        named_bar_sync(1, kNWC * 32);
#pragma unroll
        for (int k = 0; k < (G * kNWC + 31) / 32; ++k) {
            const int idx = k * 32 + lane;
            const int h = idx / kNWC, ww = idx % kNWC;
            float mx = h < G ? wmax[(bpar * kNWC + ww) * 8 + h] : -INFINITY;
#pragma unroll
            for (int o = kNWC / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
                if (hh / (32 / kNWC) == k) mbN[hh] = __shfl_sync(0xffffffffu, mx, (hh % (32 / kNWC)) * kNWC);
        }
        bpar ^= 1;
        // ---- weights and this warp's block sums
#pragma unroll
        for (int k = 0; k < (G * RW + 31) / 32; ++k) {
            const int idx = k * 32 + lane;
            const int h = idx / RW, rl = idx % RW;
            float mbh = 0.f;
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
                if (hh == h) mbh = mbN[hh];
            const float s = h < G ? scr[h * RW + rl] : -INFINITY;
            const float pw = s == -INFINITY ? 0.f : exp2f(s - mbh);
            float sum = pw;
#pragma unroll
            for (int o = RW / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (h < G) scr[h * RW + rl] = pw;
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
                if (hh / (32 / RW) == k) lbN[hh] = __shfl_sync(0xffffffffu, sum, (hh % (32 / RW)) * RW);
        }
        __syncwarp();

        // ---- P.V of this warp's rows
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < E2; ++e) tN[h][e] = 0ull;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int rl = i * RPW + half;
            const int r = w * RW + rl;
            if (r < nvalid) {
                uint64_t v2[E2];
                E::template load_pairs<C::CB>(sV + (size_t)r * C::ROWB + ch * C::CB, v2);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float pw = scr[h * RW + rl];
                    const uint64_t p2 = pk2(pw, pw);
#pragma unroll
                    for (int e = 0; e < E2; ++e) tN[h][e] = fma2(p2, v2[e], tN[h][e]);
                }
            }
        }
        release();  // K, V and q of this slot are no longer read

        if (kART) {
            // probe partials of this lane's rows: slot rank = probe columns before it
            const int vb = v & 1;
            float* pp = part + (((size_t)vb * kNWC + w) * RPW + half) * C::PST;
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                if ((my_mask >> e) & 1u) {
                    const int s = my_base + __popc(my_mask & ((1u << e) - 1u));
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float lo, hi;
                        up2(tN[h][e >> 1], lo, hi);
                        pp[s * C::GP + h] = (e & 1) ? hi : lo;
                    }
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h) plb[(vb * kNWC + w) * G + h] = lbN[h];
            }
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h) pmb[(vb * kNWC + w) * G + h] = mbN[h];
            }
            const int vN = publish(mt);
            if (LAG) {
                if (pending) {
                    const int d = wait_dec(vP);
                    if (d < 0) return;
                    fold(tP, mbP, lbP);
                    pending = false;
                    if (d == kStop) {
                        if (!epilogue(mP.b, mP.g)) return;
                        reset();
                        stopped_item = mP.item;
                        if (mt.item == mP.item) {  // computed past the stop: wait for its discard
                            if (wait_dec(vN) < 0) return;
                            advance();
                            continue;
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    mbP[h] = mbN[h];
                    lbP[h] = lbN[h];
#pragma unroll
                    for (int e = 0; e < E2; ++e) tP[h][e] = tN[h][e];
                }
                mP = mt;
                vP = vN;
                pending = true;
                if (mt.pos == mt.n - 1 && !resolve_pending()) return;  // the last listed block
            } else {
                const int d = wait_dec(vN);
                if (d < 0) return;
                fold(tN, mbN, lbN);
                if (d == kStop) {
                    if (!epilogue(mt.b, mt.g)) return;
                    reset();
                    stopped_item = mt.item;
                }
            }
        } else {
            fold(tN, mbN, lbN);
            if (mt.pos == mt.n - 1) {
                if (!epilogue(mt.b, mt.g)) return;
                reset();
                stopped_item = mt.item;
            }
        }
        advance();
    }
}


// ---------------------------------------------------------------------------
// tensor-core consumer warps (bf16), in NG groups of GW warps. Group k takes
// ring entries u = k, k + NG, ... of the same stream of items, so NG blocks of
// one item are in flight at once; each group keeps its own partial
// accumulators, and when an item ends the groups merge them together.
//
// Warp wg of a group owns keys 16 wg .. 16 wg + 15 of a block.
// S^T (16 keys x 8 heads) = K (16 x d) . Q^T (d x 8) with mma.m16n8k16, K and
// Q^T fragments by ldmatrix from 128B-swizzled tiles; the weights are split
// into bf16 hi + lo parts (p = hi + lo to ~2^-17) and
// O^T (d x 8 heads) += V^T (d x 16 keys) . P^T (16 keys x 8 heads), V^T
// fragments by ldmatrix.trans, P^T fragments by movmatrix of the S^T layout.
// Heads beyond G are carried as zeros.
//
// Every entry gives the statistics warp one record (a computed block, or a
// block / pad / failed / empty entry without data), in entry order. A group
// publishes the record of its current entry, then waits for the decision on
// its previous entry: "continue" folds that block into the group's
// accumulators, "stop" folds it and ends the item, "discard" (a block past a
// stop) ends the item without folding. A group also ends its item when its
// next entry belongs to another item.
// ---------------------------------------------------------------------------
template <class C, bool kART>
__device__ void consumer_tc(const Params& p, unsigned char* ring, const SlotMeta* meta, uint64_t* full,
                            uint64_t* empty, uint64_t* part_full, uint64_t* dec_bar, uint64_t* cbar, const Layout& L,
                            unsigned char* smem, const int* prank, Ctrl* ctrl) {
    constexpr int G = C::GQ, D = C::DD, KS = C::KS, NWC = C::NWC, GW = C::GW, NG = C::NG, NB = C::NB;
    using E = typename C::E;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = w / GW, wg = w % GW;  // group, warp within the group
    const int grp = lane >> 2, tig = lane & 3;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    const bool v0 = h0 < G, v1 = h1 < G;  // the score columns of this lane hold real heads
    // the O^T columns of this lane: heads (q0, q1); with the split tile, lanes with
    // tig >= 2 hold the low parts of heads 2 tig - 4, 2 tig - 3
    constexpr bool SPLITN = C::SPLITN;
    const bool lo_lane = SPLITN && tig >= 2;
    const int q0 = lo_lane ? h0 - 4 : h0, q1 = q0 + 1;
    const bool u0 = q0 < G, u1 = q1 < G;          // columns that belong to a real head
    const bool w0 = u0 && !lo_lane, w1 = u1 && !lo_lane;  // ... and are written by this lane
    float* part = reinterpret_cast<float*>(smem + L.part);
    float* plb = reinterpret_cast<float*>(smem + L.plb);
    float* pmb = reinterpret_cast<float*>(smem + L.pmb);
    float* eacc = reinterpret_cast<float*>(smem + L.eacc);
    unsigned char* sQt = smem + L.qt + (size_t)gi * 8 * C::ROWB;
    const uint32_t qtbase = smem_addr(sQt);
    const float scale = 1.4426950408889634f / sqrtf((float)D);
    const int ctid = threadIdx.x;   // 0 .. NWC*32-1
    const int gtid = ctid % (GW * 32);
    const int gbar = 1 + gi;        // named barrier of the group
    // this lane's O^T rows are d = 16 mt + grp + 8 r; bit 2 mt + r marks a probe column,
    // byte 2 mt + r of prk holds its rank among the probe columns
    uint32_t pbits = 0;
    uint32_t prk[(2 * KS + 3) / 4];
#pragma unroll
    for (int i = 0; i < (2 * KS + 3) / 4; ++i) prk[i] = 0;
    if (kART) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rk = prank[16 * mt + grp + 8 * r];
                if (rk >= 0) {
                    pbits |= 1u << (2 * mt + r);
                    prk[(2 * mt + r) >> 2] |= (uint32_t)rk << (8 * ((2 * mt + r) & 3));
                }
            }
    }
    const int mi = lane >> 3, lr = lane & 7;
    const int keyK = wg * 16 + (mi & 1) * 8 + lr;   // K rows for the S^T A fragments
    const int chK = mi >> 1;
    const int keyV = wg * 16 + (mi >> 1) * 8 + lr;  // V rows for the O^T A fragments
    const int chV = mi & 1;
    // K / V tiles: pages of PR rows one after another, each as [column half][PR rows][128 B],
    // 16-byte chunks of a row XOR-swizzled by the row (128B swizzle)
    const int PR = p.Ps < kBK ? p.Ps : kBK;
    const int lpr = 31 - __clz(PR);
    auto rowoff = [=](int row) -> uint32_t {
        return (uint32_t)(((row >> lpr) * (C::ROWB / 128) * PR + (row & (PR - 1))) * 128);
    };
    auto sw = [=](uint32_t base, int row, int chunk) -> uint32_t {
        return base + rowoff(row) + (uint32_t)((chunk >> 3) * PR * 128 + (((chunk & 7) ^ (row & 7)) << 4));
    };

    float acc[KS][4], tN[KS][4], tP[KS][4];
    float mrun[2], lrun[2], mbN[2], lbN[2], mbP[2], lbP[2];
    auto reset = [&]() {
#pragma unroll
        for (int j = 0; j < 2; ++j) { mrun[j] = -INFINITY; lrun[j] = 0.f; }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][c] = 0.f;
    };
    reset();
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) tN[mt][c] = tP[mt][c] = 0.f;
    mbN[0] = mbN[1] = mbP[0] = mbP[1] = lbN[0] = lbN[1] = lbP[0] = lbP[1] = 0.f;

    int u = gi;            // this group's current ring entry (= its record number)
    uint32_t cbph = 0;     // phase of the all-consumer barrier
    int cur_item = -1, curb = 0, curg = 0;  // the item held in this group's accumulators
    int stopped_item = -1;                  // the last item this group ended
    bool pending = false, pcomp = false;    // previous entry awaiting its decision; computed?
    int uP = 0, itemP = -1, posP = 0, nP = 0;

    auto cbar_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(cbar);
        const bool r = wait_bounded<C::HINT>(cbar, cbph, ctrl, p.hdr, 111 + gi);
        cbph ^= 1u;
        return r;
    };
    auto out_index = [&](int b, int g, int h, int col) -> size_t {
        return ((size_t)b * p.Hq + (size_t)g * G + h) * D + col;
    };
    auto wait_dec = [&](int rec) -> int {
        if (!wait_bounded<C::HINT>(&dec_bar[rec % NB], (uint32_t)(rec / NB) & 1u, ctrl, p.hdr, 121 + gi)) return -1;
        return ctrl->dec[rec % NB];
    };
    auto fold = [&](const float (&t)[KS][4], const float* mb, const float* lb) {
        float a[2], bb[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const bool none = mb[j] == -INFINITY;  // a head beyond G, or no valid key: keep the state
            const float mn = none ? mrun[j] : fmaxf(mrun[j], mb[j]);
            a[j] = none ? 1.f : exp2f(mrun[j] - mn);
            bb[j] = none ? 0.f : exp2f(mb[j] - mn);
            lrun[j] = none ? lrun[j] : a[j] * lrun[j] + bb[j] * lb[j];
            mrun[j] = mn;
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][c] = a[c & 1] * acc[mt][c] + bb[c & 1] * t[mt][c];
    };
    // both groups together: merge the per-warp partials of the item (each group
    // has its own running maxima) and write O = sum / weight sum
    auto finalize = [&]() -> bool {
        float* mine = eacc + (size_t)w * (G * D + 2 * G);
        if constexpr (SPLITN) {
            // high + low parts (both lanes carry the same running max and sum)
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[mt][c] += __shfl_xor_sync(0xffffffffu, acc[mt][c], 2);
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int d = 16 * mt + grp + 8 * r;
                if (w0) mine[q0 * D + d] = acc[mt][2 * r];
                if (w1) mine[q1 * D + d] = acc[mt][2 * r + 1];
            }
        if (grp == 0) {
            if (w0) { mine[G * D + q0] = lrun[0]; mine[G * D + G + q0] = mrun[0]; }
            if (w1) { mine[G * D + q1] = lrun[1]; mine[G * D + G + q1] = mrun[1]; }
        }
        if (!cbar_sync()) return false;
        const int ob = curb, og = curg;  // both groups hold the same item
        const bool okbg = ob >= 0 && ob < p.B && og >= 0 && og < p.Hkv;
        if (!okbg && ctid == 0) record_check(p.hdr, 3, ob, og, u);
        for (int idx = ctid; idx < G * D; idx += NWC * 32) {
            const int h = idx / D;
            float mx = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < NWC; ++ww) mx = fmaxf(mx, eacc[(size_t)ww * (G * D + 2 * G) + G * D + G + h]);
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int ww = 0; ww < NWC; ++ww) {
                const float* e = eacc + (size_t)ww * (G * D + 2 * G);
                const float mw = e[G * D + G + h];
                const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
                num += f * e[idx];
                den += f * e[G * D + h];
            }
            if (okbg) E::store(p.out, out_index(ob, og, h, idx - h * D), num / den);
        }
        return cbar_sync();
    };
    auto write_zero = [&](int b, int g) {
        if (b < 0 || b >= p.B || g < 0 || g >= p.Hkv) {
            if (gtid == 0) record_check(p.hdr, 4, b, g, u);
            return;
        }
        for (int idx = gtid; idx < G * D; idx += GW * 32) E::store(p.out, out_index(b, g, idx / D, idx % D), 0.f);
    };
    // the record of entry u for the statistics warp
    auto publish = [&](const SlotMeta& mt, int kind, bool computed) {
        const int rb = u % NB;
        if (kART) {
            if (computed) {
                // probe partial rows: one per warp, two (high, low) with the split tile;
                // predicated stores, no divergent branches
                float* pp = part + (((size_t)rb * GW + wg) * C::PRW + (lo_lane ? 1 : 0)) * C::PST + q0;
#pragma unroll
                for (int m = 0; m < KS; ++m)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const bool on = (pbits >> (2 * m + r)) & 1u;
                        const int rank = (int)((prk[(2 * m + r) >> 2] >> (8 * ((2 * m + r) & 3))) & 0xffu);
                        float* dst = pp + rank * C::GP;
                        if (G >= 2) st_shared_if(on && u1, dst, tN[m][2 * r], tN[m][2 * r + 1]);
                        if (G % 2) st_shared_if(on && u0 && !u1, dst, tN[m][2 * r]);
                    }
                st_shared_if(grp == 0 && w0, &plb[(rb * GW + wg) * G + (w0 ? q0 : 0)], lbN[0]);
                st_shared_if(grp == 0 && w1, &plb[(rb * GW + wg) * G + (w1 ? q1 : 0)], lbN[1]);
                st_shared_if(grp == 0 && w0, &pmb[(rb * GW + wg) * G + (w0 ? q0 : 0)], mbN[0]);
                st_shared_if(grp == 0 && w1, &pmb[(rb * GW + wg) * G + (w1 ? q1 : 0)], mbN[1]);
            }
            if (wg == 0 && lane == 0) {
                SlotMeta& r = ctrl->info[rb];
                r.kind = kind; r.item = mt.item; r.pos = mt.pos; r.n = mt.n; r.c = mt.c; r.has0 = mt.has0;
            }
            __syncwarp();
            mbar_arrive_if(lane == 0, &part_full[rb]);
        }
    };

    for (;;) {
        const int slot = u % p.stages;
        if (NG > 1 && u >= p.stages) {
            // the slot's previous entry belongs to another group and its copies may land
            // after this group's own earlier entries: wait until it has been consumed, so
            // that the parity test below cannot match that older fill
            if (!wait_bounded<C::HINT>(&empty[slot], (uint32_t)(u / p.stages - 1) & 1u, ctrl, p.hdr, 151 + gi)) return;
        }
        if (!wait_bounded<C::HINT>(&full[slot], (uint32_t)(u / p.stages) & 1u, ctrl, p.hdr, 101 + gi)) return;
        SlotMeta mt = meta[slot];
        if (mt.kind < 0 || mt.kind > kSlotPad ||
            (mt.kind == kSlotBlock && (mt.item < 0 || mt.item >= p.num_items || mt.nvalid < 1 || mt.nvalid > kBK ||
                                       mt.pos < 0 || mt.pos >= mt.n || mt.b < 0 || mt.b >= p.B || mt.g < 0 ||
                                       mt.g >= p.Hkv))) {
            if (lane == 0) record_check(p.hdr, 5, u, mt.kind, mt.item);
            mt.kind = kSlotPad;
            mt.item = -2;
        }
        const bool is_data = mt.kind == kSlotBlock || mt.kind == kSlotPad;
        const bool compute = mt.kind == kSlotBlock && mt.item != stopped_item;
        if (compute) {
            unsigned char* sK = ring + (size_t)slot * C::SLOT;
            unsigned char* sV = sK + C::KVB;
            if (mt.pos < NG) {
                // the item's queries into this group's swizzled 8-row area (rows past G zero),
                // once every warp of the group has finished the previous item's scores
                named_bar_sync(gbar, GW * 32);
                const unsigned char* sQ = sK + 2 * C::KVB;
                constexpr int QCH = 8 * (C::ROWB / 16);
                for (int i = gtid; i < QCH; i += GW * 32) {
                    const int row = i / (C::ROWB / 16), c = i % (C::ROWB / 16);
                    const uint4 val = row < G ? *reinterpret_cast<const uint4*>(sQ + (size_t)row * C::ROWB + c * 16)
                                              : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(sQt + (c >> 3) * 1024 + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = val;
                }
                named_bar_sync(gbar, GW * 32);
            }
            const int nvalid = mt.nvalid;
            // ---- S^T for this warp's 16 keys (two independent accumulation chains);
            // ldmatrix / mma.sync / movmatrix are warp-aligned: reconverge before them
            float s4[4] = {0.f, 0.f, 0.f, 0.f}, s4b[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t kbase = smem_addr(sK), vbase = smem_addr(sV);
            __syncwarp();
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
                uint32_t b00, b01, b10, b11;
                {
                    const int c = 4 * kp + mi;
                    ldsm_x4(qtbase + (uint32_t)((c >> 3) * 1024 + lr * 128 + (((c & 7) ^ lr) << 4)), b00, b01, b10, b11);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ks = 2 * kp + h;
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(sw(kbase, keyK, 2 * ks + chK), a0, a1, a2, a3);
                    mma_bf16(h ? s4b : s4, a0, a1, a2, a3, h ? b10 : b00, h ? b11 : b01);
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) s4[c] += s4b[c];
            const int k0 = wg * 16 + grp, k1 = k0 + 8;
            float sc[4];
            sc[0] = (k0 < nvalid && v0) ? s4[0] * scale : -INFINITY;
            sc[1] = (k0 < nvalid && v1) ? s4[1] * scale : -INFINITY;
            sc[2] = (k1 < nvalid && v0) ? s4[2] * scale : -INFINITY;
            sc[3] = (k1 < nvalid && v1) ? s4[3] * scale : -INFINITY;
            // ---- this warp's block max per head (each warp keeps its own running max;
            // the statistics warp and the item's final merge rescale between warps)
            float mb0 = fmaxf(sc[0], sc[2]), mb1 = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                mb0 = fmaxf(mb0, __shfl_xor_sync(0xffffffffu, mb0, o));
                mb1 = fmaxf(mb1, __shfl_xor_sync(0xffffffffu, mb1, o));
            }
            float pw[4];
            pw[0] = sc[0] == -INFINITY ? 0.f : exp2f(sc[0] - mb0);
            pw[1] = sc[1] == -INFINITY ? 0.f : exp2f(sc[1] - mb1);
            pw[2] = sc[2] == -INFINITY ? 0.f : exp2f(sc[2] - mb0);
            pw[3] = sc[3] == -INFINITY ? 0.f : exp2f(sc[3] - mb1);
            float l0 = pw[0] + pw[2], l1 = pw[1] + pw[3];
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            }
            uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
            if constexpr (SPLITN) {
                // low-part lanes take the weights, maxima and sums of lane ^ 2
                float px[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) px[c] = __shfl_xor_sync(0xffffffffu, pw[c], 2);
                const float mx0 = __shfl_xor_sync(0xffffffffu, mb0, 2), mx1 = __shfl_xor_sync(0xffffffffu, mb1, 2);
                const float lx0 = __shfl_xor_sync(0xffffffffu, l0, 2), lx1 = __shfl_xor_sync(0xffffffffu, l1, 2);
                float t[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) t[c] = lo_lane ? px[c] : pw[c];
                mbN[0] = lo_lane ? mx0 : mb0; mbN[1] = lo_lane ? mx1 : mb1;
                lbN[0] = lo_lane ? lx0 : l0; lbN[1] = lo_lane ? lx1 : l1;
                const uint32_t hA = pack_bf16(t[0], t[1]), hB = pack_bf16(t[2], t[3]);
                const uint32_t lA = pack_bf16(t[0] - bf16_lo_f(hA), t[1] - bf16_hi_f(hA));
                const uint32_t lB = pack_bf16(t[2] - bf16_lo_f(hB), t[3] - bf16_hi_f(hB));
                __syncwarp();
                bh0 = movm_t(lo_lane ? lA : hA);
                bh1 = movm_t(lo_lane ? lB : hB);
            } else {
                mbN[0] = mb0; mbN[1] = mb1; lbN[0] = l0; lbN[1] = l1;
                // ---- P^T fragments: hi and lo bf16 parts, transposed by movmatrix
                const uint32_t hA = pack_bf16(pw[0], pw[1]), hB = pack_bf16(pw[2], pw[3]);
                const uint32_t lA = pack_bf16(pw[0] - bf16_lo_f(hA), pw[1] - bf16_hi_f(hA));
                const uint32_t lB = pack_bf16(pw[2] - bf16_lo_f(hB), pw[3] - bf16_hi_f(hB));
                __syncwarp();
                bh0 = movm_t(hA); bh1 = movm_t(hB); bl0 = movm_t(lA); bl1 = movm_t(lB);
            }
            // ---- rows past the sequence end hold stale data: zero this warp's, so 0 * V stays 0
            if (nvalid < wg * 16 + 16) {
                const int r0 = max(nvalid, wg * 16);
                const int nchunks = (wg * 16 + 16 - r0) * (C::ROWB / 16);
                for (int i = lane; i < nchunks; i += 32) {
                    const int row = r0 + i / (C::ROWB / 16), c = i % (C::ROWB / 16);
                    *reinterpret_cast<uint4*>(sV + rowoff(row) + (c >> 3) * PR * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- O^T partial of this block
            __syncwarp();
#pragma unroll
            for (int m = 0; m < KS; ++m) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(sw(vbase, keyV, 2 * m + chV), a0, a1, a2, a3);
                tN[m][0] = tN[m][1] = tN[m][2] = tN[m][3] = 0.f;
                mma_bf16(tN[m], a0, a1, a2, a3, bh0, bh1);
                if constexpr (!SPLITN) mma_bf16(tN[m], a0, a1, a2, a3, bl0, bl1);
            }
        }
        __syncwarp();
        mbar_arrive_if(lane == 0 && mt.kind != kSlotEnd, &empty[slot]);  // the slot's data are no longer read

        // ---- this entry's record, then the decision on the previous one
        publish(mt, (mt.kind == kSlotBlock && !compute) ? kSlotPad : mt.kind, compute);
        bool ended = false;
        if (pending) {
            int d;
            if (kART) {
                d = wait_dec(uP);
                if (d < 0) return;
            } else {
                d = !pcomp ? kDiscard : (posP == nP - 1 ? kStop : kContinue);
            }
            if (pcomp && d != kDiscard) fold(tP, mbP, lbP);
            ended = (d == kStop || d == kDiscard) && itemP == cur_item;
            pending = false;
        }
        if (cur_item != -1 && (ended || mt.item != cur_item || !is_data)) {
            if (!finalize()) return;
            reset();
            stopped_item = cur_item;
            cur_item = -1;
        }
        if (mt.kind == kSlotEnd) return;
        if (!is_data && mt.pos == 0) write_zero(mt.b, mt.g);
        if (is_data && cur_item == -1 && mt.item != stopped_item) {
            cur_item = mt.item;
            curb = mt.b;
            curg = mt.g;
        }
        // this entry waits for its decision until this group's next entry
        pending = true;
        pcomp = compute;
        uP = u;
        itemP = mt.item;
        posP = mt.pos;
        nP = mt.n;
        if (compute) {
#pragma unroll
            for (int m = 0; m < KS; ++m)
#pragma unroll
                for (int c = 0; c < 4; ++c) tP[m][c] = tN[m][c];
            mbP[0] = mbN[0]; mbP[1] = mbN[1]; lbP[0] = lbN[0]; lbP[1] = lbN[1];
        }
        u += NG;
    }
}

// ---------------------------------------------------------------------------
// tensor-core consumers (bf16), head dims split between the warps of a group
//
// A group of GW warps takes one 64-key block per ring entry. Warp wg computes
// the scores of keys 16 wg .. 16 wg + 15 (S^T = K Q^T with mma.m16n8k16 from
// the swizzled tiles) and its weights p = 2^(s - e) against its own max
// rounded up to an integer e, so that two warps' weights differ by an exact
// power of two. The warps exchange their weights (as P^T mma fragments),
// exponents and weight sums through shared memory (one named barrier per
// block); then warp wg computes O^T for head dims wg*DW .. (wg+1)*DW - 1 over
// all 64 keys, each key chunk's fragment scaled to the group max exactly (a
// bf16 multiply by a power of two). The weights are split into bf16 high +
// low parts (p = hi + lo to ~2^-17); for G <= 4 the two parts share one 8-column
// tile (columns 4-7 hold the low parts). Every warp therefore holds the
// complete block result for its dims, and each probe column has one writer.
//
// Every entry gives the statistics warp one record (a computed block, or a
// block / pad / failed / empty entry without data), in entry order. A group
// publishes the record of its current entry, then waits for the decision on
// its previous entry: "continue" folds that block into the group's
// accumulators, "stop" folds it and ends the item, "discard" (a block past a
// stop) ends the item without folding. A group also ends its item when its
// next entry belongs to another item.
// ---------------------------------------------------------------------------
template <class C, bool kART>
__device__ void consumer_ds(const Params& p, unsigned char* ring, const SlotMeta* meta, uint64_t* full,
                            uint64_t* empty, uint64_t* part_full, uint64_t* dec_bar, uint64_t* cbar, const Layout& L,
                            unsigned char* smem, const int* prank, Ctrl* ctrl) {
    constexpr int G = C::GQ, D = C::DD, KS = C::KS, NWC = C::NWC, GW = C::GW, NG = C::NG, NB = C::NB;
    constexpr int DW = C::DW, MT = C::MT, XBW = C::XBW;
    using E = typename C::E;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = w / GW, wg = w % GW;  // group, warp within the group
    const int grp = lane >> 2, tig = lane & 3;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    const bool v0 = h0 < G, v1 = h1 < G;  // the score columns of this lane hold real heads
    // the O^T columns of this lane: heads (q0, q1); with the split tile, lanes with
    // tig >= 2 hold the low parts of heads 2 tig - 4, 2 tig - 3
    constexpr bool SPLITN = C::SPLITN;
    const bool lo_lane = SPLITN && tig >= 2;
    const int q0 = lo_lane ? h0 - 4 : h0, q1 = q0 + 1;
    const bool u0 = q0 < G, u1 = q1 < G;                  // columns that belong to a real head
    const bool w0 = u0 && !lo_lane, w1 = u1 && !lo_lane;  // ... and are written by this lane
    // the head of this lane's P^T fragment column (column grp)
    const int hb = (SPLITN && grp >= 4) ? grp - 4 : grp;
    float* part = reinterpret_cast<float*>(smem + L.part);
    float* plb = reinterpret_cast<float*>(smem + L.plb);
    float* pmb = reinterpret_cast<float*>(smem + L.pmb);
    float* eacc = reinterpret_cast<float*>(smem + L.eacc);
    uint32_t* xb = reinterpret_cast<uint32_t*>(smem + L.xb + (size_t)gi * C::XGB);
    float* xm = reinterpret_cast<float*>(xb + 2 * GW * 32 * XBW);
    float* xl = xm + 2 * 8 * GW;
    unsigned char* sQt = smem + L.qt + (size_t)gi * 8 * C::ROWB;
    const uint32_t qtbase = smem_addr(sQt);
    const float scale = 1.4426950408889634f / sqrtf((float)D);
    const int ctid = threadIdx.x;   // 0 .. NWC*32-1
    const int gtid = ctid % (GW * 32);
    const int gbar = 1 + gi;        // named barrier of the group
    // this lane's O^T rows are d = wg DW + 16 mt + 8 r + grp; bit 2 mt + r marks a probe
    // column, byte 2 mt + r of prk holds its rank among the probe columns
    // ... and pofs[2 mt + r] the byte offset of its slot in a record's partial rows
    uint32_t pbits = 0;
    uint32_t pofs[2 * MT];
#pragma unroll
    for (int k = 0; k < 2 * MT; ++k) pofs[k] = 0;
    if (kART) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int rk = prank[wg * DW + 16 * mt + 8 * r + grp];
                if (rk >= 0 && u0) {
                    pbits |= 1u << (2 * mt + r);
                    pofs[2 * mt + r] = (uint32_t)(((lo_lane ? C::PST : 0) + q0 + rk * C::GP) * 4);
                }
            }
    }
    const uint32_t part_base = smem_addr(part);
    const int mi = lane >> 3, lr = lane & 7;
    const int keyK = wg * 16 + (mi & 1) * 8 + lr;  // K rows for the S^T A fragments
    const int chK = mi >> 1;
    const int keyV = (mi >> 1) * 8 + lr;           // V rows (within a 16-key chunk) for the O^T A fragments
    const int chV = mi & 1;
    // K / V tiles: pages of PR rows one after another, each as [column half][PR rows][128 B],
    // 16-byte chunks of a row XOR-swizzled by the row (128B swizzle)
    const int PR = p.Ps < kBK ? p.Ps : kBK;
    const int lpr = 31 - __clz(PR);
    auto rowoff = [=](int row) -> uint32_t {
        return (uint32_t)(((row >> lpr) * (C::ROWB / 128) * PR + (row & (PR - 1))) * 128);
    };
    auto sw = [=](uint32_t base, int row, int chunk) -> uint32_t {
        return base + rowoff(row) + (uint32_t)((chunk >> 3) * PR * 128 + (((chunk & 7) ^ (row & 7)) << 4));
    };

    float acc[MT][4], tN[MT][4], tP[MT][4];
    float mrun[2], lrun[2], mbN[2], lbN[2], mbP[2], lbP[2];
    auto reset = [&]() {
#pragma unroll
        for (int j = 0; j < 2; ++j) { mrun[j] = -INFINITY; lrun[j] = 0.f; }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][c] = 0.f;
    };
    reset();
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) tN[mt][c] = tP[mt][c] = 0.f;
    mbN[0] = mbN[1] = mbP[0] = mbP[1] = lbN[0] = lbN[1] = lbP[0] = lbP[1] = 0.f;

    int u = gi;            // this group's current ring entry (= its record number)
    int xpar = 0;          // exchange buffer of the next computed block
    uint32_t cbph = 0;     // phase of the all-consumer barrier
    int cur_item = -1, curb = 0, curg = 0;  // the item held in this group's accumulators
    int stopped_item = -1;                  // the last item this group ended
    bool pending = false, pcomp = false;    // previous entry awaiting its decision; computed?
    int uP = 0, itemP = -1, posP = 0, nP = 0;

    auto cbar_sync = [&]() -> bool {
        __syncwarp();
        mbar_arrive_if(lane == 0, cbar);
        const bool r = wait_bounded<C::HINT>(cbar, cbph, ctrl, p.hdr, 111 + gi);
        cbph ^= 1u;
        return r;
    };
    auto out_index = [&](int b, int g, int h, int col) -> size_t {
        return ((size_t)b * p.Hq + (size_t)g * G + h) * D + col;
    };
    auto wait_dec = [&](int rec) -> int {
        if (!wait_bounded<C::HINT>(&dec_bar[rec % NB], (uint32_t)(rec / NB) & 1u, ctrl, p.hdr, 121 + gi)) return -1;
        return ctrl->dec[rec % NB];
    };
    auto fold = [&](const float (&t)[MT][4], const float* mb, const float* lb) {
        float a[2], bb[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const bool none = mb[j] == -INFINITY;  // a head beyond G, or no valid key: keep the state
            const float mn = none ? mrun[j] : fmaxf(mrun[j], mb[j]);
            a[j] = none ? 1.f : exp2f(mrun[j] - mn);
            bb[j] = none ? 0.f : exp2f(mb[j] - mn);
            lrun[j] = none ? lrun[j] : a[j] * lrun[j] + bb[j] * lb[j];
            mrun[j] = mn;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][c] = a[c & 1] * acc[mt][c] + bb[c & 1] * t[mt][c];
    };
    // write O = sum / weight sum for this warp's dims; with several groups, merge the
    // groups' partials (each has its own running maxima) through shared memory first
    auto finalize = [&]() -> bool {
        if constexpr (SPLITN) {
            // high + low parts (both lanes carry the same running max and sum)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[mt][c] += __shfl_xor_sync(0xffffffffu, acc[mt][c], 2);
        }
        const int ob = curb, og = curg;  // every group holds the same item
        const bool okbg = ob >= 0 && ob < p.B && og >= 0 && og < p.Hkv;
        if constexpr (NG == 1) {
            if (!okbg) {
                if (lane == 0) record_check(p.hdr, 3, ob, og, u);
                return true;
            }
            const float r0 = 1.f / lrun[0], r1 = 1.f / lrun[1];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int d = wg * DW + 16 * mt + 8 * r + grp;
                    if (w0) E::store(p.out, out_index(ob, og, q0, d), acc[mt][2 * r] * r0);
                    if (w1) E::store(p.out, out_index(ob, og, q1, d), acc[mt][2 * r + 1] * r1);
                }
            return true;
        } else {
            float* mine = eacc + (size_t)gi * (C::XGB / 4);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int d = wg * DW + 16 * mt + 8 * r + grp;
                    if (w0) mine[q0 * D + d] = acc[mt][2 * r];
                    if (w1) mine[q1 * D + d] = acc[mt][2 * r + 1];
                }
            if (wg == 0 && grp == 0) {
                if (w0) { mine[G * D + q0] = lrun[0]; mine[G * D + G + q0] = mrun[0]; }
                if (w1) { mine[G * D + q1] = lrun[1]; mine[G * D + G + q1] = mrun[1]; }
            }
            if (!cbar_sync()) return false;
            if (!okbg && ctid == 0) record_check(p.hdr, 3, ob, og, u);
            for (int idx = ctid; idx < G * D; idx += NWC * 32) {
                const int h = idx / D;
                float mx = -INFINITY;
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) mx = fmaxf(mx, eacc[(size_t)gg * (C::XGB / 4) + G * D + G + h]);
                float num = 0.f, den = 0.f;
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) {
                    const float* e = eacc + (size_t)gg * (C::XGB / 4);
                    const float mw = e[G * D + G + h];
                    const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
                    num += f * e[idx];
                    den += f * e[G * D + h];
                }
                if (okbg) E::store(p.out, out_index(ob, og, h, idx - h * D), num / den);
            }
            return cbar_sync();
        }
    };
    auto write_zero = [&](int b, int g) {
        if (b < 0 || b >= p.B || g < 0 || g >= p.Hkv) {
            if (gtid == 0) record_check(p.hdr, 4, b, g, u);
            return;
        }
        for (int idx = gtid; idx < G * D; idx += GW * 32) E::store(p.out, out_index(b, g, idx / D, idx % D), 0.f);
    };
    // the record of entry u for the statistics warp
    auto publish = [&](const SlotMeta& mt, int kind, bool computed) {
        const int rb = u % NB;
        if (kART) {
            if (computed) {
                // probe partial rows (high and low parts with the split tile); predicated
                // stores, no divergent branches
                const uint32_t rec = part_base + (uint32_t)(rb * C::PRW * C::PST * 4);
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const bool on = (pbits >> (2 * m + r)) & 1u;
                        if (G >= 2) st_shared_if(on && u1, rec + pofs[2 * m + r], tN[m][2 * r], tN[m][2 * r + 1]);
                        if (G % 2) st_shared_if(on && !u1, rec + pofs[2 * m + r], tN[m][2 * r]);
                    }
                const bool lead = wg == 0 && grp == 0;
                st_shared_if(lead && w0, &plb[rb * G + (w0 ? q0 : 0)], lbN[0]);
                st_shared_if(lead && w1, &plb[rb * G + (w1 ? q1 : 0)], lbN[1]);
                st_shared_if(lead && w0, &pmb[rb * G + (w0 ? q0 : 0)], mbN[0]);
                st_shared_if(lead && w1, &pmb[rb * G + (w1 ? q1 : 0)], mbN[1]);
            }
            if (wg == 0 && lane == 0) {
                SlotMeta& r = ctrl->info[rb];
                r.kind = kind; r.item = mt.item; r.pos = mt.pos; r.n = mt.n; r.c = mt.c; r.has0 = mt.has0;
            }
            __syncwarp();
            mbar_arrive_if(lane == 0, &part_full[rb]);
        }
    };
    // bf16x2 multiplier 2^(e - emax) for a power-of-two exponent difference (0 below bf16 range)
    auto pow2_bf16x2 = [](float e, float emax) -> uint32_t {
        const float d = e - emax;  // an integer <= 0, or NaN / -inf
        const int k = d >= -126.f ? (int)d : -1000;
        const uint32_t bits = k >= -126 ? (uint32_t)(k + 127) << 7 : 0u;
        return bits | (bits << 16);
    };

    for (;;) {
        const int slot = u % p.stages;
        if (NG > 1 && u >= p.stages) {
            // the slot's previous entry belongs to another group and its copies may land
            // after this group's own earlier entries: wait until it has been consumed, so
            // that the parity test below cannot match that older fill
            if (!wait_bounded<C::HINT>(&empty[slot], (uint32_t)(u / p.stages - 1) & 1u, ctrl, p.hdr, 151 + gi)) return;
        }
        if (!wait_bounded<C::HINT>(&full[slot], (uint32_t)(u / p.stages) & 1u, ctrl, p.hdr, 101 + gi)) return;
        SlotMeta mt = meta[slot];
        if (mt.kind < 0 || mt.kind > kSlotPad ||
            (mt.kind == kSlotBlock && (mt.item < 0 || mt.item >= p.num_items || mt.nvalid < 1 || mt.nvalid > kBK ||
                                       mt.pos < 0 || mt.pos >= mt.n || mt.b < 0 || mt.b >= p.B || mt.g < 0 ||
                                       mt.g >= p.Hkv))) {
            if (lane == 0) record_check(p.hdr, 5, u, mt.kind, mt.item);
            mt.kind = kSlotPad;
            mt.item = -2;
        }
        const bool is_data = mt.kind == kSlotBlock || mt.kind == kSlotPad;
        const bool compute = mt.kind == kSlotBlock && mt.item != stopped_item;
        if (compute) {
            unsigned char* sK = ring + (size_t)slot * C::SLOT;
            unsigned char* sV = sK + C::KVB;
            if (mt.pos < NG) {
                // the item's queries into this group's swizzled 8-row area (rows past G zero),
                // once every warp of the group has finished the previous item's scores
                named_bar_sync(gbar, GW * 32);
                const unsigned char* sQ = sK + 2 * C::KVB;
                constexpr int QCH = 8 * (C::ROWB / 16);
                for (int i = gtid; i < QCH; i += GW * 32) {
                    const int row = i / (C::ROWB / 16), c = i % (C::ROWB / 16);
                    const uint4 val = row < G ? *reinterpret_cast<const uint4*>(sQ + (size_t)row * C::ROWB + c * 16)
                                              : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(sQt + (c >> 3) * 1024 + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = val;
                }
                named_bar_sync(gbar, GW * 32);
            }
            const int nvalid = mt.nvalid;
            // ---- S^T for this warp's 16 keys (two independent accumulation chains);
            // ldmatrix / mma.sync / movmatrix are warp-aligned: reconverge before them
            float s4[4] = {0.f, 0.f, 0.f, 0.f}, s4b[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t kbase = smem_addr(sK), vbase = smem_addr(sV);
            __syncwarp();
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
                uint32_t b00, b01, b10, b11;
                {
                    const int c = 4 * kp + mi;
                    ldsm_x4(qtbase + (uint32_t)((c >> 3) * 1024 + lr * 128 + (((c & 7) ^ lr) << 4)), b00, b01, b10, b11);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ks = 2 * kp + h;
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(sw(kbase, keyK, 2 * ks + chK), a0, a1, a2, a3);
                    mma_bf16(h ? s4b : s4, a0, a1, a2, a3, h ? b10 : b00, h ? b11 : b01);
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) s4[c] += s4b[c];
            const int k0 = wg * 16 + grp, k1 = k0 + 8;
            float sc[4];
            sc[0] = (k0 < nvalid && v0) ? s4[0] * scale : -INFINITY;
            sc[1] = (k0 < nvalid && v1) ? s4[1] * scale : -INFINITY;
            sc[2] = (k1 < nvalid && v0) ? s4[2] * scale : -INFINITY;
            sc[3] = (k1 < nvalid && v1) ? s4[3] * scale : -INFINITY;
            // ---- this warp's max per head over its keys, rounded up to an integer exponent
            float e0 = fmaxf(sc[0], sc[2]), e1 = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                e0 = fmaxf(e0, __shfl_xor_sync(0xffffffffu, e0, o));
                e1 = fmaxf(e1, __shfl_xor_sync(0xffffffffu, e1, o));
            }
            e0 = ceilf(e0);
            e1 = ceilf(e1);
            float pw[4];
            pw[0] = sc[0] == -INFINITY ? 0.f : exp2f(sc[0] - e0);
            pw[1] = sc[1] == -INFINITY ? 0.f : exp2f(sc[1] - e1);
            pw[2] = sc[2] == -INFINITY ? 0.f : exp2f(sc[2] - e0);
            pw[3] = sc[3] == -INFINITY ? 0.f : exp2f(sc[3] - e1);
            float l0 = pw[0] + pw[2], l1 = pw[1] + pw[3];
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            }
            // ---- P^T fragments of this warp's keys: hi and lo bf16 parts, transposed by movmatrix
            uint32_t bf[XBW];
            if constexpr (SPLITN) {
                // low-part lanes take the weights of lane ^ 2
                float px[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) px[c] = __shfl_xor_sync(0xffffffffu, pw[c], 2);
                float t[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) t[c] = lo_lane ? px[c] : pw[c];
                const uint32_t hA = pack_bf16(t[0], t[1]), hB = pack_bf16(t[2], t[3]);
                const uint32_t lA = pack_bf16(t[0] - bf16_lo_f(hA), t[1] - bf16_hi_f(hA));
                const uint32_t lB = pack_bf16(t[2] - bf16_lo_f(hB), t[3] - bf16_hi_f(hB));
                __syncwarp();
                bf[0] = movm_t(lo_lane ? lA : hA);
                bf[1] = movm_t(lo_lane ? lB : hB);
            } else {
                const uint32_t hA = pack_bf16(pw[0], pw[1]), hB = pack_bf16(pw[2], pw[3]);
                const uint32_t lA = pack_bf16(pw[0] - bf16_lo_f(hA), pw[1] - bf16_hi_f(hA));
                const uint32_t lB = pack_bf16(pw[2] - bf16_lo_f(hB), pw[3] - bf16_hi_f(hB));
                __syncwarp();
                bf[0] = movm_t(hA); bf[1] = movm_t(hB); bf[2] = movm_t(lA); bf[3] = movm_t(lB);
            }
            // ---- publish fragments, exponents and sums to the group (every head column,
            // -inf / 0 for heads past G), then wait for the other warps of the group
            uint32_t* xbp = xb + (size_t)xpar * GW * 32 * XBW;
            float* xmp = xm + xpar * 8 * GW;
            float* xlp = xl + xpar * 8 * GW;
            if constexpr (XBW == 2)
                *reinterpret_cast<uint2*>(xbp + ((size_t)wg * 32 + lane) * 2) = make_uint2(bf[0], bf[1]);
            else
                *reinterpret_cast<uint4*>(xbp + ((size_t)wg * 32 + lane) * 4) = make_uint4(bf[0], bf[1], bf[2], bf[3]);
            st_shared_if(grp == 0, &xmp[h0 * GW + wg], e0);
            st_shared_if(grp == 0, &xmp[h1 * GW + wg], e1);
            st_shared_if(grp == 0, &xlp[h0 * GW + wg], l0);
            st_shared_if(grp == 0, &xlp[h1 * GW + wg], l1);
            // ---- rows past the sequence end hold stale data: zero this warp's dims of them,
            // so that 0 * V stays 0
            if (nvalid < kBK) {
                constexpr int CPR = DW / 8;  // 16-byte chunks of a row in this warp's dims
                const int nchunks = (kBK - nvalid) * CPR;
                for (int i = lane; i < nchunks; i += 32) {
                    const int row = nvalid + i / CPR, c = wg * CPR + i % CPR;
                    *reinterpret_cast<uint4*>(sV + rowoff(row) + (c >> 3) * PR * 128 + (((c & 7) ^ (row & 7)) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            named_bar_sync(gbar, GW * 32);
            // ---- the group's max exponent and weight sum per head
            float emx[2], ebh = -INFINITY;
            {
                const float4 mq0 = *reinterpret_cast<const float4*>(xmp + (u0 ? q0 : 0) * GW);
                const float4 mq1 = *reinterpret_cast<const float4*>(xmp + (u1 ? q1 : 0) * GW);
                const float4 lq0 = *reinterpret_cast<const float4*>(xlp + (u0 ? q0 : 0) * GW);
                const float4 lq1 = *reinterpret_cast<const float4*>(xlp + (u1 ? q1 : 0) * GW);
                static_assert(GW == 4, "one float4 per head");
                emx[0] = fmaxf(fmaxf(mq0.x, mq0.y), fmaxf(mq0.z, mq0.w));
                emx[1] = fmaxf(fmaxf(mq1.x, mq1.y), fmaxf(mq1.z, mq1.w));
                auto wsum = [](const float4& m, const float4& l, float mx) {
                    float s = 0.f;
                    s += m.x == -INFINITY ? 0.f : exp2f(m.x - mx) * l.x;
                    s += m.y == -INFINITY ? 0.f : exp2f(m.y - mx) * l.y;
                    s += m.z == -INFINITY ? 0.f : exp2f(m.z - mx) * l.z;
                    s += m.w == -INFINITY ? 0.f : exp2f(m.w - mx) * l.w;
                    return s;
                };
                mbN[0] = u0 ? emx[0] : -INFINITY;
                mbN[1] = u1 ? emx[1] : -INFINITY;
                lbN[0] = u0 && emx[0] != -INFINITY ? wsum(mq0, lq0, emx[0]) : 0.f;
                lbN[1] = u1 && emx[1] != -INFINITY ? wsum(mq1, lq1, emx[1]) : 0.f;
            }
            const float4 mb4 = *reinterpret_cast<const float4*>(xmp + hb * GW);
            ebh = fmaxf(fmaxf(mb4.x, mb4.y), fmaxf(mb4.z, mb4.w));
            const float mbw[4] = {mb4.x, mb4.y, mb4.z, mb4.w};
            // ---- O^T of this warp's dims over the block's 64 keys, chunk by chunk
#pragma unroll
            for (int m = 0; m < MT; ++m) tN[m][0] = tN[m][1] = tN[m][2] = tN[m][3] = 0.f;
            __syncwarp();
#pragma unroll
            for (int c = 0; c < GW; ++c) {
                uint32_t b[XBW];
                if constexpr (XBW == 2) {
                    const uint2 t2 = *reinterpret_cast<const uint2*>(xbp + ((size_t)c * 32 + lane) * 2);
                    b[0] = t2.x; b[1] = t2.y;
                } else {
                    const uint4 t4 = *reinterpret_cast<const uint4*>(xbp + ((size_t)c * 32 + lane) * 4);
                    b[0] = t4.x; b[1] = t4.y; b[2] = t4.z; b[3] = t4.w;
                }
                const uint32_t sc2 = hb < G ? pow2_bf16x2(mbw[c], ebh) : 0u;
#pragma unroll
                for (int k = 0; k < XBW; ++k) b[k] = hmul2_bf16(b[k], sc2);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(sw(vbase, 16 * c + keyV, 2 * (wg * MT + m) + chV), a0, a1, a2, a3);
                    mma_bf16(tN[m], a0, a1, a2, a3, b[0], b[1]);
                    if constexpr (!SPLITN) mma_bf16(tN[m], a0, a1, a2, a3, b[2], b[3]);
                }
            }
            xpar ^= 1;
        }
        __syncwarp();
        mbar_arrive_if(lane == 0 && mt.kind != kSlotEnd, &empty[slot]);  // the slot's data are no longer read

        // ---- this entry's record, then the decision on the previous one
        publish(mt, (mt.kind == kSlotBlock && !compute) ? kSlotPad : mt.kind, compute);
        bool ended = false;
        if (pending) {
            int d;
            if (kART) {
                d = wait_dec(uP);
                if (d < 0) return;
            } else {
                d = !pcomp ? kDiscard : (posP == nP - 1 ? kStop : kContinue);
            }
            if (pcomp && d != kDiscard) fold(tP, mbP, lbP);
            ended = (d == kStop || d == kDiscard) && itemP == cur_item;
            pending = false;
        }
        if (cur_item != -1 && (ended || mt.item != cur_item || !is_data)) {
            if (!finalize()) return;
            reset();
            stopped_item = cur_item;
            cur_item = -1;
        }
        if (mt.kind == kSlotEnd) return;
        if (!is_data && mt.pos == 0) write_zero(mt.b, mt.g);
        if (is_data && cur_item == -1 && mt.item != stopped_item) {
            cur_item = mt.item;
            curb = mt.b;
            curg = mt.g;
        }
        // this entry waits for its decision until this group's next entry
        pending = true;
        pcomp = compute;
        uP = u;
        itemP = mt.item;
        posP = mt.pos;
        nP = mt.n;
        if (compute) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int c = 0; c < 4; ++c) tP[m][c] = tN[m][c];
            mbP[0] = mbN[0]; mbP[1] = mbN[1]; lbP[0] = lbN[0]; lbP[1] = lbN[1];
        }
        u += NG;
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// tensor cores: one group per CTA runs two CTAs per SM; two to four groups one
template <class C>
struct MinBlocks {
    static constexpr int value = (C::TC && C::NG == 1) ? 2 : 1;
};

template <class C, bool kART>
__global__ void __launch_bounds__(C::THREADS, (MinBlocks<C>::value))
    art_decode_kernel(const Params p, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
    constexpr int NWC = C::NWC;
    constexpr int D = C::DD;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzled tiles need a 1024-byte aligned ring
    unsigned char* smem = smem_raw;
    if (C::TC) smem += (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    const Layout L = make_layout<C>(p.stages);
    unsigned char* ring = smem;
    SlotMeta* meta = reinterpret_cast<SlotMeta*>(smem + L.meta);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + p.stages;
    uint64_t* part_full = empty + p.stages;
    uint64_t* dec_bar = part_full + C::NB;
    uint64_t* cbar = dec_bar + C::NB;
    uint64_t* stall_bar = cbar + 1;  // never completed (the failure-path test hook)
    uint64_t* jobb = stall_bar + 1;  // copy warps: [stages] job posted
    SlotJob* job = reinterpret_cast<SlotJob*>(smem + L.job);
    int* last_entry = reinterpret_cast<int*>(job + p.stages);
    int* pmask = reinterpret_cast<int*>(smem + L.ptab);
    int* pbase = pmask + C::LPR;
    int* prank = pbase + C::LPR;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + L.ctrl);

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::GW);  // an entry is consumed by one group
        }
        for (int b = 0; b < C::NB; ++b) {
            mbar_init(&part_full[b], C::GW);
            mbar_init(&dec_bar[b], 1);
            ctrl->dec[b] = 0;
        }
        mbar_init(cbar, NWC);
        mbar_init(stall_bar, 1);
        if (C::COPYW)
            for (int s = 0; s < p.stages; ++s) {
                mbar_init(&jobb[s], 1);
                last_entry[s] = -1;
            }
        ctrl->stop_item = -1;
        ctrl->abort = 0;
        ctrl->wait_ns = p.wait_ns;
        fence_mbar_init();
    }
    if (tid < C::LPR) {
        // probe columns of chunk `tid`, and the probe entries with a smaller column
        uint32_t mask = 0;
        int base = 0;
        if (kART && p.probe) {
            for (int k = 0; k < p.m; ++k) {
                const int col = __ldg(&p.probe[k]);
                const int off = col - tid * C::EPC;
                if (off >= 0 && off < C::EPC) mask |= 1u << off;
                if (col >= 0 && col < tid * C::EPC) ++base;
            }
        }
        pmask[tid] = (int)mask;
        pbase[tid] = base;
    }
    if (tid < D) {
        // rank of column `tid` among the probe columns, or -1
        int found = 0, rank = 0;
        if (kART && p.probe) {
            for (int k = 0; k < p.m; ++k) {
                const int col = __ldg(&p.probe[k]);
                if (col == tid) found = 1;
                if (col >= 0 && col < tid) ++rank;
            }
        }
        prank[tid] = found ? rank : -1;
    }
    if (C::TC && tid == (NWC + 2) * 32) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tv)) : "memory");
    }
    __syncthreads();

    const int warp = tid >> 5;
    if (p.stall && warp < NWC && !wait_bounded(stall_bar, 0u, ctrl, p.hdr, 161)) return;
    if (warp == NWC) {
        producer_warp<C, kART>(p, ring, meta, job, full, empty, jobb, ctrl, &tk, &tv);
    } else if (warp == NWC + 1) {
        if (kART)
            stat_warp<C>(p, reinterpret_cast<const float*>(smem + L.part), reinterpret_cast<const float*>(smem + L.plb),
                         reinterpret_cast<const float*>(smem + L.pmb), reinterpret_cast<float*>(smem + L.sh),
                         part_full, dec_bar, ctrl);
    } else if (warp >= NWC + 2) {  // the copy warps (none without COPYW)
        if constexpr (C::COPYW) copy_warp<C>(p, ring, job, last_entry, full, jobb, ctrl, &tk, &tv, warp - (NWC + 2));
    } else if constexpr (C::TC) {
        if constexpr (C::DS)
            consumer_ds<C, kART>(p, ring, meta, full, empty, part_full, dec_bar, cbar, L, smem, prank, ctrl);
        else
            consumer_tc<C, kART>(p, ring, meta, full, empty, part_full, dec_bar, cbar, L, smem, prank, ctrl);
    } else {
        consumer_warps<C, kART>(p, ring, meta, full, empty, part_full, dec_bar, cbar, L, smem, pmask, pbase, ctrl);
    }
}

// Largest ring depth (2..8 slots) that lets `want` CTAs share one SM.
template <class C>
inline int pick_stages(int want, int smem_per_sm, int smem_per_block) {
    for (int s = 8; s >= 2; --s) {
        const size_t t = make_layout<C>(s).total;
        if ((int)t <= smem_per_block && (size_t)want * (t + 1024) <= (size_t)smem_per_sm) return s;
    }
    return 0;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// A 2-D bf16 view [rows = pages * Hkv * page_size][D] of a cache, read in
// boxes of 64 columns (128 bytes) by min(page_size, 64) rows, 128B-swizzled.
// A 3-D bf16 view {64 columns, rows, column halves} of the same cache (strides: a row
// D * 2 bytes, a half 128 bytes), read one page of rows (both halves) per copy: the box
// lands as [half][rows][64 columns], 128B-swizzled.
inline cudaError_t make_cache_map3(CUtensorMap* m, const void* base, long long rows, int D, int Ps) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)(Ps < kBK ? Ps : kBK), (cuuint32_t)(D / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

inline cudaError_t make_cache_map(CUtensorMap* m, const void* base, long long rows, int D, int Ps) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(Ps < kBK ? Ps : kBK)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <class C, bool kART>
cudaError_t launch_variant(Params p, cudaStream_t stream, int force_stages, LaunchInfo* li, int sms, int smem_sm,
                           int smem_blk) {
    constexpr int D = C::DD;
    auto kern = art_decode_kernel<C, kART>;
    cudaError_t e;
    // several CTAs per SM only pay when there are items for them
    const int per_sm = (p.num_items + sms - 1) / sms;
    const int want = MinBlocks<C>::value < per_sm ? MinBlocks<C>::value : per_sm;
    int stages = force_stages >= 2 && force_stages <= 8 ? force_stages : pick_stages<C>(want, smem_sm, smem_blk);
    if (stages == 0) stages = pick_stages<C>(1, smem_sm, smem_blk);
    if constexpr (C::NCW > 1) stages -= stages % C::NCW;  // every slot's entries go to one copy warp
    // At an item's end each group merges while it holds the slot of its first entry of
    // the next item, so all NG such entries must fit in the ring at once.
    constexpr int kMinStages = C::NG < 2 ? 2 : (C::NCW > 1 ? (C::NG + C::NCW - 1) / C::NCW * C::NCW : C::NG);
    if (stages < kMinStages) stages = kMinStages;
    const size_t smem = make_layout<C>(stages).total;
    if ((int)smem > smem_blk) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    int occ = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::THREADS, smem)) != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof tk);
    std::memset(&tv, 0, sizeof tv);
    if (C::TC) {
        const long long rows = (long long)p.num_pages * p.Hkv * p.Ps;
        if (rows >= (1LL << 31)) return cudaErrorInvalidValue;
        // one copy per page where the driver takes the 3-D view, else one per column half
        const char* env3 = std::getenv("ART_TMA3D");
        p.tma3d = (!env3 || std::atoi(env3) != 0) && make_cache_map3(&tk, p.k, rows, D, p.Ps) == cudaSuccess &&
                  make_cache_map3(&tv, p.v, rows, D, p.Ps) == cudaSuccess;
        if (!p.tma3d) {
            if ((e = make_cache_map(&tk, p.k, rows, D, p.Ps)) != cudaSuccess) return e;
            if ((e = make_cache_map(&tv, p.v, rows, D, p.Ps)) != cudaSuccess) return e;
        }
    }
    p.stages = stages;
    int grid = sms * occ;
    if (grid > p.num_items) grid = p.num_items;
    if (li) { li->grid = grid; li->stages = stages; li->smem = smem; li->ctas_per_sm = occ; }
    kern<<<grid, C::THREADS, smem, stream>>>(p, tk, tv);
    return cudaGetLastError();
}

template <bool kBF16, int D, int G, bool kART>
cudaError_t launch_main(Params p, cudaStream_t stream, int force_stages, LaunchInfo* li) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 0, smem_sm = 0, smem_blk = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    // bf16: one CTA per SM with three consumer groups (head dims split) that take
    // alternate blocks of an item. Measured against one group and two CTAs per SM (keys
    // split): 15 % faster on the ragged batch, 3 % on the paged one, and the statistics
    // cost 8 % instead of 15-20 %; the last item on an SM then also runs three blocks at a
    // time. With no more items than SMs each CTA runs one item, whose blocks the consumer
    // groups bound: four groups then (3 % faster on 128 items of 512 blocks; with more
    // items, three groups and their deeper ring are 7 % faster). ART_GROUPS (1..4)
    // overrides the choice.
    const char* env = std::getenv("ART_GROUPS");
    const int groups = env ? std::atoi(env) : (p.num_items <= sms ? 4 : 3);
    if constexpr (kBF16) {
        // a probe over more than kMaxProbe columns per head (up to every head dim): one
        // group of four warps with the head dims split, so that each probe column has one
        // writer and three records of probe rows fit in shared memory
        if constexpr (kART)
            if (p.m > kMaxProbe)
                return launch_variant<Cfg<true, D, G, 1, true, D>, kART>(p, stream, force_stages, li, sms, smem_sm,
                                                                           smem_blk);
        if (groups == 2)
            return launch_variant<Cfg<kBF16, D, G, 2>, kART>(p, stream, force_stages, li, sms, smem_sm, smem_blk);
        if (groups == 3)
            return launch_variant<Cfg<kBF16, D, G, 3>, kART>(p, stream, force_stages, li, sms, smem_sm, smem_blk);
        if (groups == 4)
            return launch_variant<Cfg<kBF16, D, G, 4>, kART>(p, stream, force_stages, li, sms, smem_sm, smem_blk);
    }
    return launch_variant<Cfg<kBF16, D, G, 1>, kART>(p, stream, force_stages, li, sms, smem_sm, smem_blk);
}

}  // namespace art

#define ART_INSTANTIATE(BF, D, G)                                                                           \
    template cudaError_t art::launch_main<BF, D, G, true>(art::Params, cudaStream_t, int, art::LaunchInfo*); \
    template cudaError_t art::launch_main<BF, D, G, false>(art::Params, cudaStream_t, int, art::LaunchInfo*);
