// art_units.cuh -- ART decode attention with one item spread over many CTAs.
//
// With fewer items (sequence b, KV head g) than SMs, one CTA per item leaves
// most SMs idle, and an item runs no faster than one SM streams. Here each
// item's visit list is cut into units of `ck` consecutive entries that any CTA
// may take:
//
//   plan        numbers the units round by round (unit k of every item, longest
//               lists first, before unit k + 1 of any item), then ck fix pieces
//               per item; CTAs claim units in that order from a counter.
//   producer    TMA copies of a unit's blocks into the ring of shared-memory
//               slots, and of the unit's queries into one of two query tiles.
//   consumers   softmax attention of each block for the G query heads (tensor
//               cores, one group of 4 warps with the head dims split, as in the
//               one-CTA kernel's default groups), folded into the unit's partial
//               output (every warp: the same running max and weight sum, the
//               output sums of its dims), which goes to global memory at the
//               unit's end; each block's probe partials go to the summary warp.
//   summary     announces each unit to the test warp when its first block's
//               record arrives, turns each block's probe partials into a block
//               summary (max, weight sum, probe sums per head), stored per CTA
//               in global memory, and publishes the unit's probe aggregate.
//   tests       takes the state of the probe before the unit from a look-back
//               over the item's earlier units (their aggregates, back to the
//               nearest one that has published its inclusive state), as soon as
//               the unit is announced, while its blocks are still computed.
//               Once the unit is summarized it runs the stability test of
//               each block of the unit in order, exactly as one pass over the
//               list would (ART paper sec. 3.2; explainer sec. 2.2-2.4), and
//               publishes the unit's stable bits. With patience <= ck the
//               patience count entering a unit depends on the previous unit's
//               bits only, so the unit can name its first stop position (if
//               any) at once and lowers the item's stop to it (atomicMin).
//               Every position before the one-pass stop sees the same
//               statistics as the one-pass rule, so the smallest position named
//               is that stop.
//   fix pieces  ck per item, claimed after every unit: once every unit up to
//               the one holding the item's stop has named its stop (or been
//               skipped), piece j recomputes
//               block j of the stopping unit if it lies at or before the stop
//               (that unit's own partial also holds blocks after it), one block
//               per CTA, so the recompute is spread over the GPU.
//   combine     a second kernel (programmatic dependent launch) merges, per
//               item and query head, the partials of the units before the
//               stopping unit and of the fix pieces (or the stopping unit itself
//               when it ends at the stop): O = sums / weight sums, in a fixed
//               order.
//
// A unit whose item has already stopped before it when it is claimed is
// skipped; units claimed before the stop was known are read and discarded.
//
// The dense twin (kART = false) runs the same units without the statistics:
// the plan sets every item's stop to its last block, no fix pieces exist, and
// the merge combines all units.
//
// A CTA waits on another CTA's unit only for a unit claimed earlier; every CTA
// works through its units in claim order and the compute of a unit never
// waits on another unit, so the waits end. They are bounded all the same.
#pragma once

#include <cstddef>

#include "art_kernel.cuh"

namespace art {

constexpr int kUnitBlocks = 16;     // ck: ART blocks per unit at most
constexpr int kUnitMinBlocks = 8;   // ... and at least (the workspace is sized for it)
constexpr int kUnitRecs = 5;        // block records in flight from the consumers to the statistics warp
constexpr size_t kUnitMaxWsBytes = (size_t)4 << 30;  // the unit path's workspace area at most
constexpr int kUnitMaxCtas = 512;   // unit-kernel CTAs at most (each has its own summary store)
constexpr int kUnitMaxK = 4096;     // units per item at most
constexpr int kUnitWords = 10;      // words per lane of a probe state: max, weight sum, 8 probe slots

// Global-memory flags between CTAs: release stores, acquire loads (GPU scope).
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// orders this thread's earlier memory accesses before its later ones, GPU scope
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// atomic add with release semantics: this thread's earlier writes are visible first
__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Byte offsets of the unit path's workspace area (after the one-CTA path's).
struct UnitWs {
    size_t p0, stop_min, resolved, fail, ulist, tflag, uflags, agg, incl, part_o, part_ml, fix_o, fix_ml, ustore,
        total;
};

// Partials are merged over the CTA's warps before they are written: per unit (and per
// fix piece) G*D output sums [head][dim], then 16 words: the max of each head (words
// 0..7) and its weight sum (words 8..15).
constexpr int kUnitMlWords = 16;

__host__ __device__ inline UnitWs make_unit_ws(int items, int maxk, int D, int G) {
    UnitWs w;
    const size_t U = (size_t)items * maxk;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    w.p0 = take((size_t)items * 4);
    w.stop_min = take((size_t)items * 4);
    w.resolved = take((size_t)items * 4);
    w.fail = take((size_t)items * 4);
    w.ulist = take(U * 8);
    w.tflag = take(U * 4);
    w.uflags = take(U * 16);
    w.agg = take(U * 32 * kUnitWords * 4);
    w.incl = take(U * 32 * kUnitWords * 4);
    w.part_o = take(U * (size_t)G * D * 4);
    w.part_ml = take(U * kUnitMlWords * 4);
    w.fix_o = take((size_t)items * kUnitBlocks * G * D * 4);
    w.fix_ml = take((size_t)items * kUnitBlocks * kUnitMlWords * 4);
    w.ustore = take((size_t)kUnitMaxCtas * 2 * kUnitBlocks * kUnitWords * 32 * 4);
    w.total = o;
    return w;
}

struct UParams {
    const int2* ulist;  // claim position -> (item, unit index k)
    const int* p0;      // per item: list position of logical block 0, or -1
    int* stop_min;      // per item: smallest stop position named so far
    int* resolved;      // per item: units whose stop is named (or that were skipped)
    int* fail;          // per item: a page check failed in this path
    int* tflag;         // per (item, k): 1 aggregate, 2 and inclusive state, 3 skipped
    int* uflags;        // per (item, k): {stable bits, blocks, state (1 set, 3 skipped), resolved (1)}
    float* agg;         // per (item, k): [kUnitWords][32 lanes] probe state of the unit's blocks
    float* incl;        // per (item, k): the same through the unit (from the list's start)
    float* part_o;      // per (item, k): [G][D] output sums, merged over the warps
    float* part_ml;     // per (item, k): max of each head (words 0..7), weight sum (words 8..15)
    float* fix_o;       // per (item, fix piece): the piece's partial, same layout
    float* fix_ml;
    float* ustore;      // per CTA: [2][kUnitBlocks][kUnitWords][32 lanes] block summaries of the units being
                        // handed from the summary warp to the test warp (two in turn)
    int ck;             // ART blocks per unit (the kernels take it from the workspace header)
    int maxk;           // units per item at most
};

enum UnitKind : int { kUBlock = 0, kUFix = 1, kUEnd = 2 };

struct UMeta {
    int kind, item, k, j, nj, pos, n, c, nvalid, b, g, pad;
};

struct URec {
    int kind, item, k, j, nj, pad0, pad1, pad2;
};

template <int D, int G>
struct UCfg {
    using C = Cfg<true, D, G, 1, true>;  // one group of four warps, head dims split
    static constexpr int THREADS = 7 * 32;  // 4 consumer warps, producer, block summaries, tests
    static constexpr int W = C::SPL + 2;
    // a ring slot holds one block's K and V; the unit's queries go to their own tiles
    static constexpr int SLOT = 2 * C::KVB;
    static constexpr int QTB = 8 * C::ROWB;  // bytes of one query tile (8 rows, heads past G masked)
    static_assert(W <= kUnitWords, "probe state fits the workspace words");
};

struct ULayout {
    size_t meta, bars, part, plb, pmb, qt, xb, ptab, rinfo, uhdr, ctrl, total;
};

template <int D, int G>
__host__ __device__ inline ULayout make_ulayout(int stages) {
    using C = typename UCfg<D, G>::C;
    ULayout L;
    size_t o = (size_t)stages * UCfg<D, G>::SLOT;
    L.meta = o;
    o += (size_t)stages * sizeof(UMeta);
    o = align_up(o, 16);
    L.bars = o;  // full[stages], empty[stages], part_full[NB], part_empty[NB]
    o += (size_t)(2 * stages + 2 * kUnitRecs + 9) * sizeof(uint64_t);  // ... ufull[2], uempty[2], stall, qfree[2], ustart[2]
    o = align_up(o, 16);
    static_assert(C::DS && C::RGW == 1, "one writer per probe column");
    L.part = o;  // [NB][PRW][PST] probe partial rows (one writer per column)
    o += (size_t)kUnitRecs * C::PRW * C::PST * sizeof(float);
    L.plb = o;  // [NB][G] block weight sums
    o += (size_t)kUnitRecs * G * sizeof(float);
    L.pmb = o;  // [NB][G] block maxima (integer exponents)
    o += (size_t)kUnitRecs * G * sizeof(float);
    o = align_up(o, 1024);
    L.qt = o;  // two tiles of a unit's queries, 8 rows (heads past G masked), 128B-swizzled by the copy
    o += (size_t)2 * UCfg<D, G>::QTB;
    o = align_up(o, 16);
    L.xb = o;  // [2 block parities][4 warps][32 lanes] P^T fragments, then [2][8][4] exponents,
               // then [2][8][4] weight sums
    o += (size_t)C::XGB;
    L.ptab = o;  // rank of each head dim among the probe dims, or -1
    o += (size_t)D * sizeof(int);
    o = align_up(o, 16);
    L.rinfo = o;
    o += (size_t)kUnitRecs * sizeof(URec);
    o = align_up(o, 16);
    L.uhdr = o;  // [2]: the units of the two summary buffers, then [2]: the units started in them
    o += 4 * sizeof(URec);
    o = align_up(o, 16);
    L.ctrl = o;  // only the abort and stop_item words of a Ctrl are used here
    static_assert(offsetof(Ctrl, abort) + sizeof(int) <= 128 && offsetof(Ctrl, stop_item) + sizeof(int) <= 128 &&
                      offsetof(Ctrl, wait_ns) + sizeof(unsigned long long) <= 128,
                  "the words of Ctrl used by the unit kernel fit its 128 bytes");
    o += 128;
    L.total = align_up(o, 128) + 1024;  // room to align the ring to 1024 bytes
    return L;
}

// Polls a global flag until it is >= want (the value read goes to `got`);
// false when this CTA gave up elsewhere or after its wait limit. Every lane
// then loads the flag once more with acquire semantics, so each lane's later
// loads of the payload are ordered after it.
__device__ __forceinline__ bool poll_flag(const int* flag, int want, int& got, Ctrl* ctrl, WsHeader* hdr,
                                          int where) {
    const int lane = threadIdx.x & 31;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0;; ++it) {
        int v = 0;
        if (lane == 0) v = ld_acquire_gpu(flag);
        v = __shfl_sync(0xffffffffu, v, 0);
        if (v >= want) {
            got = ld_acquire_gpu(flag);
            got = __shfl_sync(0xffffffffu, got, 0);
            return true;
        }
        int quit = 0;
        if (lane == 0) {
            if (ld_volatile_shared(&ctrl->abort)) quit = 1;
            else if ((it & 63u) == 63u && global_ns() - t0 > ctrl->wait_ns) {
                st_volatile_shared(&ctrl->abort, 1);
                atomicOr(&hdr->status, ART_STATUS_TIMEOUT);
                record_check(hdr, where, want, v, 0);
                quit = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, quit, 0)) return false;
        __nanosleep(64);
    }
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <class C, class UC>
__device__ void producer_u(const Params& p, const UParams& up, unsigned char* ring, UMeta* meta, uint64_t* full,
                           uint64_t* empty, uint64_t* qfree, unsigned char* qt, Ctrl* ctrl, const CUtensorMap* tk,
                           const CUtensorMap* tv, const CUtensorMap* tq) {
    constexpr int G = C::GQ;
    constexpr int NH = C::ROWB / 128;
    const int lane = threadIdx.x & 31;
    int slot = 0;
    uint32_t round = 0;
    unsigned long long issued = 0;
    bool ok = true;
    int uloc = 0;  // units of this CTA with blocks issued (selects the query tile)
    const int n_reg = p.hdr->n_regular, n_units = p.hdr->n_units;  // written by the plan kernel

    auto acquire = [&]() -> bool { return wait_bounded(&empty[slot], (round & 1u) ^ 1u, ctrl, p.hdr, 231); };
    auto advance = [&]() {
        ++issued;
        if (++slot == p.stages) {
            slot = 0;
            ++round;
        }
    };
    // a unit that will not be computed: mark it for the look-backs and the stop count
    auto mark_skipped = [&](int item, int k) {
        const size_t iu = (size_t)item * up.maxk + k;
        if (lane == 0) {
            st_release_gpu(&up.tflag[iu], 3);
            st_release_gpu(&up.uflags[4 * iu + 2], 3);
            st_release_gpu(&up.uflags[4 * iu + 3], 1);
            red_release_add(&up.resolved[item], 1);
        }
        __syncwarp();
    };
    // Waits (bounded) until the item's stop is final and returns it: once every unit up to
    // the one holding the smallest position named so far has been resolved, no unit can
    // name a smaller one (later units start past it). Units after the stop need not have
    // finished. Returns false on abort or timeout.
    auto final_stop = [&](int item, int n, int& t_out) -> bool {
        const unsigned long long t0 = global_ns();
        for (unsigned it = 0;; ++it) {
            int t = 0;
            if (lane == 0) t = ld_acquire_gpu(&up.stop_min[item]);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t >= 0 && t < n) {
                const int kk = t / up.ck;
                bool all = true;
                for (int base = 0; base <= kk && all; base += 32) {
                    const int k = base + lane;
                    const int r = k <= kk ? ld_acquire_gpu(&up.uflags[4 * ((size_t)item * up.maxk + k) + 3]) : 1;
                    all = __all_sync(0xffffffffu, r >= 1);
                }
                if (all) {
                    // a unit resolved after the first read may have named a smaller stop
                    int t2 = 0;
                    if (lane == 0) t2 = ld_acquire_gpu(&up.stop_min[item]);
                    t2 = __shfl_sync(0xffffffffu, t2, 0);
                    if (t2 == t) {
                        t_out = t;
                        return true;
                    }
                    continue;
                }
            }
            int quit = 0;
            if (lane == 0) {
                if (ld_volatile_shared(&ctrl->abort)) quit = 1;
                else if ((it & 63u) == 63u && global_ns() - t0 > ctrl->wait_ns) {
                    st_volatile_shared(&ctrl->abort, 1);
                    atomicOr(&p.hdr->status, ART_STATUS_TIMEOUT);
                    record_check(p.hdr, 232, item, t, n);
                    quit = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, quit, 0)) return false;
            __nanosleep(64);
        }
    };

    // One listed position of a unit per lane (cnt <= 32): the logical block c, its valid
    // tokens, the pages holding them (with pages larger than a block, the first row).
    struct Pos {
        int c, nvalid, npv, r0;
        int pg[8];
    };
    // the position's pages; their loads are issued here, the values first used later
    auto load_pages = [&](Pos& ps, int b, int seq_len, bool active) {
        ps.nvalid = 0;
        ps.npv = 0;
        ps.r0 = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) ps.pg[q] = 0;
        const int t0 = ps.c * kBK;
        if (!active || ps.c < 0 || t0 >= seq_len) return;
        const int32_t* trow = p.block_table + (size_t)b * p.max_pages;
        ps.nvalid = min(kBK, seq_len - t0);
        if (p.Ps <= kBK) {
            ps.npv = (ps.nvalid + p.Ps - 1) / p.Ps;
            const int pfirst = t0 / p.Ps;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < ps.npv) ps.pg[q] = trow[pfirst + q];
        } else {
            ps.npv = 1;
            ps.pg[0] = trow[t0 / p.Ps];
            ps.r0 = t0 % p.Ps;
        }
    };
    // a listed position outside the sequence or a page outside the pool
    auto pos_bad = [&](const Pos& ps, int seq_len, bool active) -> bool {
        if (!active) return false;
        if (ps.c < 0 || ps.c * kBK >= seq_len) return true;
        bool bad = false;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (q < ps.npv && (ps.pg[q] < 0 || ps.pg[q] >= p.num_pages)) bad = true;
        return bad;
    };

    // ---- the next unit is claimed and resolved in steps (claim, list entry, item, visit
    // entries, page ids), right after the current unit's last block is issued: the ring
    // still holds that many blocks for the consumers meanwhile. (Claiming a unit while the
    // current one is still being issued measured slower: a unit claimed early publishes its
    // aggregate late, and the look-backs of later units of its item wait for it.)
    int nst = 0;            // steps of the next unit done (5: resolved)
    unsigned nclaim = 0;    // lane 0: the claim, until step 1
    int nu = 0, nitem = -1, nk = 0, nb = 0, ng = 0, nn = 0, nfirst = 0, ncnt = 0, nseq = 0;
    bool nend = false, nfix = false, nok = false;  // nok: a regular unit of a known item
    int2 ne = make_int2(0, 0);
    ItemInfo ninf;
    ninf.n = 0;
    ninf.flags = 0;
    Pos np;
    np.c = 0;
    auto next_step = [&]() {
        if (nst == 0) {
            if (lane == 0) nclaim = atomicAdd(&p.hdr->uclaim, 1u);
        } else if (nst == 1) {
            nu = (int)__shfl_sync(0xffffffffu, nclaim, 0);
            nend = nu >= n_units;
            nfix = !nend && nu >= n_reg;
            if (!nend && !nfix) ne = up.ulist[nu];
        } else if (nst == 2) {
            nok = false;
            if (!nend && !nfix) {
                nitem = ne.x;
                nk = ne.y;
                if (nitem >= 0 && nitem < p.num_items) {
                    nok = true;
                    ninf = p.info[nitem];
                    nb = nitem / p.Hkv;
                    ng = nitem - nb * p.Hkv;
                    nseq = p.seq_lens[nb];
                } else if (lane == 0) {
                    record_check(p.hdr, 201, nu, nitem, 0);
                }
            }
        } else if (nst == 3) {
            if (nok) {
                nn = (ninf.flags & kItemBad) ? 0 : ninf.n;
                const int nch = (nn + up.ck - 1) / up.ck;
                if (nk < 0 || nk >= nch) {
                    if (lane == 0) record_check(p.hdr, 234, nitem, nk, nch);
                    nok = false;
                } else {
                    nfirst = nk * up.ck;
                    ncnt = min(up.ck, nn - nfirst);
                    const int32_t* vrow = p.visit ? p.visit + (size_t)nitem * p.max_visit : nullptr;
                    np.c = 0;
                    if (lane < ncnt) np.c = vrow ? vrow[nfirst + lane] : nfirst + lane;
                }
            }
        } else if (nst == 4) {
            if (nok) load_pages(np, nb, nseq, lane < ncnt);
        }
        ++nst;
    };

    // issues the blocks of a unit (lanes hold its positions)
    auto issue_unit = [&](bool fix, int item, int k, int first, int cnt, int n, int b, int g, const Pos& ps) -> bool {
        for (int j = 0; j < cnt; ++j) {
            if (!acquire()) return false;
            const int cj = __shfl_sync(0xffffffffu, ps.c, j);
            const int nvj = __shfl_sync(0xffffffffu, ps.nvalid, j);
            const int npj = __shfl_sync(0xffffffffu, ps.npv, j);
            const int r0j = __shfl_sync(0xffffffffu, ps.r0, j);
            int pgj[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) pgj[q] = __shfl_sync(0xffffffffu, ps.pg[q], j);
            const bool with_q = j == 0;
            // the unit's queries go to tile uloc % 2, once the consumers are done with the
            // unit two before it (tiles alternate between units)
            if (with_q && uloc >= 2 &&
                !wait_bounded(&qfree[uloc & 1], (uint32_t)((uloc >> 1) - 1) & 1u, ctrl, p.hdr, 235))
                return false;
            const int page_rows = p.Ps <= kBK ? p.Ps : kBK;
            const uint32_t page_bytes = (uint32_t)(page_rows * C::ROWB);
            const uint32_t bytes = 2u * npj * page_bytes + (with_q ? (uint32_t)UC::QTB : 0u);
            unsigned char* dst = ring + (size_t)slot * UC::SLOT;
            if (lane == 0) {
                UMeta& mt = meta[slot];
                mt.kind = fix ? kUFix : kUBlock; mt.item = item; mt.k = k; mt.j = j; mt.nj = cnt;
                mt.pos = first + j; mt.n = n; mt.c = cj; mt.nvalid = nvj; mt.b = b; mt.g = g;
                mbar_arrive_expect_tx(&full[slot], bytes);
            }
            __syncwarp();
            // each page's rows land as [column half][rows][128 B] (128B-swizzled), pages one
            // after another; one 3-D copy per page, or one 2-D copy per column half
            const int nop = p.tma3d ? npj : npj * NH;
            const int nbox = 2 * nop;
            const int nqc = with_q ? (p.tma3d ? 1 : NH) : 0;  // query copies: 8 rows from the group's first head
            for (int t = lane; t < nbox + nqc; t += 32) {
                if (t < nbox) {
                    const int kv = t / nop;
                    const int rem = t - kv * nop;
                    const int q = p.tma3d ? rem : rem / NH, hf = p.tma3d ? 0 : rem - (rem / NH) * NH;
                    int pk = 0;
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        if (x == q) pk = pgj[x];
                    const int y = (pk * p.Hkv + g) * p.Ps + r0j;
                    unsigned char* d = dst + kv * C::KVB + (q * NH + hf) * page_rows * 128;
                    if (p.tma3d)
                        tma_load_3d(d, kv ? tv : tk, 0, y, 0, &full[slot]);
                    else
                        tma_load_2d(d, kv ? tv : tk, hf * 64, y, &full[slot]);
                } else {
                    // rows past the group's G heads (the next group's, or zeros past the
                    // tensor) only feed score columns the consumers mask
                    unsigned char* qd = qt + (size_t)(uloc & 1) * UC::QTB;
                    const int yq = b * p.Hq + g * G;
                    if (p.tma3d)
                        tma_load_3d(qd, tq, 0, yq, 0, &full[slot]);
                    else
                        tma_load_2d(qd + (t - nbox) * 1024, tq, (t - nbox) * 64, yq, &full[slot]);
                }
            }
            __syncwarp();
            advance();
        }
        ++uloc;
        return true;
    };

    while (nst < 5) next_step();
    for (;;) {
        if (nend) {
            // nothing left to claim: the merge kernel may be launched
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            if (!acquire()) {
                ok = false;
                break;
            }
            if (lane == 0) {
                UMeta& mt = meta[slot];
                mt.kind = kUEnd; mt.item = -1; mt.k = 0; mt.j = 0; mt.nj = 1; mt.pos = 0; mt.n = 0; mt.c = -1;
                mt.nvalid = 0; mt.b = 0; mt.g = 0;
                mbar_arrive(&full[slot]);
            }
            __syncwarp();
            advance();
            break;
        }
        if (nfix) {
            // a fix piece (claimed after every regular unit): once every unit of its item has
            // named its stop, block k of the stopping unit if it lies at or before the stop
            const int f = nu - n_reg;  // fix piece f % ck of the item at claim position f / ck
            nst = 0;
            const int item = p.order[f / up.ck], k = f % up.ck;
            bool skip = item < 0 || item >= p.num_items;
            if (skip && lane == 0) record_check(p.hdr, 201, nu, item, 0);
            int first = 0, n = 0, b = 0, g = 0, seq_len = 0;
            if (!skip) {
                const ItemInfo inf = p.info[item];
                n = (inf.flags & kItemBad) ? 0 : inf.n;
                const int nch = (n + up.ck - 1) / up.ck;
                b = item / p.Hkv;
                g = item - b * p.Hkv;
                skip = nch == 0;
                int t = -1;
                if (!skip) {
                    if (!final_stop(item, n, t)) {
                        ok = false;
                        break;
                    }
                    skip = ld_acquire_gpu(&up.fail[item]) != 0;
                }
                if (!skip) {
                    if (t < 0 || t >= n) {
                        if (lane == 0) record_check(p.hdr, 233, item, t, n);
                        skip = true;
                    } else {
                        const int sfirst = t / up.ck * up.ck;
                        // the stopping unit ends at the stop, or this piece's block lies past it
                        skip = t == min(n, sfirst + up.ck) - 1 || sfirst + k > t;
                        first = sfirst + k;
                    }
                }
                if (!skip) seq_len = p.seq_lens[b];
            }
            if (!skip) {
                Pos ps;
                ps.c = 0;
                if (lane == 0) {
                    const int32_t* vrow = p.visit ? p.visit + (size_t)item * p.max_visit : nullptr;
                    ps.c = vrow ? vrow[first] : first;
                }
                load_pages(ps, b, seq_len, lane == 0);
                if (__any_sync(0xffffffffu, pos_bad(ps, seq_len, lane == 0))) {
                    if (lane == 0) {
                        atomicOr(&p.hdr->status, ART_STATUS_BAD_PAGE);
                        atomicExch(&up.fail[item], 1);
                    }
                } else if (!issue_unit(true, item, k, first, 1, n, b, g, ps)) {
                    ok = false;
                    break;
                }
            }
            while (nst < 5) next_step();
            continue;
        }
        if (!nok) {
            nst = 0;
            while (nst < 5) next_step();
            continue;
        }
        // the next unit becomes the current one
        const int item = nitem, k = nk, b = nb, g = ng, n = nn, first = nfirst, cnt = ncnt, seq_len = nseq;
        const Pos ps = np;
        const int stop_seen = ld_acquire_gpu(&up.stop_min[item]);
        nst = 0;
        if (stop_seen < first) {  // the item stopped before this unit since it was claimed
            mark_skipped(item, k);
            while (nst < 5) next_step();
            continue;
        }
        if (__any_sync(0xffffffffu, pos_bad(ps, seq_len, lane < cnt))) {
            if (lane == 0) {
                atomicOr(&p.hdr->status, ART_STATUS_BAD_PAGE);
                atomicExch(&up.fail[item], 1);
            }
            mark_skipped(item, k);
            while (nst < 5) next_step();
            continue;
        }
        if (!issue_unit(false, item, k, first, cnt, n, b, g, ps)) {
            ok = false;
            break;
        }
        while (nst < 5) next_step();
    }

    if (!ok) {
        // aborting: wait (bounded) for this CTA's own copies still in flight
        const unsigned long long lim = issued < (unsigned long long)p.stages ? issued : p.stages;
        int s = slot;
        uint32_t r = round;
        for (unsigned long long q = 0; q < lim; ++q) {
            if (--s < 0) {
                s = p.stages - 1;
                --r;
            }
            const unsigned long long t0 = global_ns();
            while (!__all_sync(0xffffffffu, mbar_try_wait(&full[s], r & 1u)) && global_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

// ---------------------------------------------------------------------------
// consumer warps: one group of four, head dims split between them.
//
// Warp wg computes the scores of keys 16 wg .. 16 wg + 15 of a block (S^T = K Q^T
// with mma.m16n8k16 from the swizzled tiles) and their weights p = 2^(s - e)
// against its own max rounded up to an integer exponent e. The four warps
// exchange the P^T fragments, exponents and weight sums through shared memory
// (one named barrier per block); warp wg then computes O^T for head dims
// wg D/4 .. (wg + 1) D/4 - 1 over all 64 keys, each key chunk's fragment scaled to
// the block's largest exponent exactly (a bf16 multiply by a power of two). The
// weights enter P.V as bf16 high + low parts (for G <= 4 both share one 8-column
// tile). Every warp so holds the same block max and weight sum per head, and each
// probe column has one writer. The block is folded into the unit's running state
// at once (no decision is waited for); at the unit's last block each warp writes
// its own dims of the unit's partial.
// ---------------------------------------------------------------------------
template <class C, class UC, bool kART>
__device__ void consumer_u(const Params& p, const UParams& up, unsigned char* ring, const UMeta* meta,
                           uint64_t* full, uint64_t* empty, uint64_t* part_full, uint64_t* part_empty,
                           uint64_t* qfree, URec* rinfo, const ULayout& L, unsigned char* smem, const int* prank,
                           Ctrl* ctrl) {
    constexpr int G = C::GQ, D = C::DD, KS = C::KS, GW = C::GW, NB = kUnitRecs;
    constexpr int DW = C::DW, MT = C::MT, XBW = C::XBW;
    constexpr bool SPLITN = C::SPLITN;
    static_assert(C::DS && GW == 4, "four warps, head dims split");
    const int wg = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 2, tig = lane & 3;
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
    const bool v0 = h0 < G, v1 = h1 < G;  // the score columns of this lane hold real heads
    // O^T columns of this lane: heads (q0, q1); with the split tile, lanes with tig >= 2
    // hold the low parts of heads 2 tig - 4, 2 tig - 3
    const bool lo_lane = SPLITN && tig >= 2;
    const int q0 = lo_lane ? h0 - 4 : h0, q1 = q0 + 1;
    const bool u0 = q0 < G, u1 = q1 < G;
    const bool w0 = u0 && !lo_lane, w1 = u1 && !lo_lane;
    const int hb = (SPLITN && grp >= 4) ? grp - 4 : grp;  // the head of this lane's P^T fragment column
    float* plb = reinterpret_cast<float*>(smem + L.plb);
    float* pmb = reinterpret_cast<float*>(smem + L.pmb);
    uint32_t* xb = reinterpret_cast<uint32_t*>(smem + L.xb);
    float* xm = reinterpret_cast<float*>(xb + 2 * GW * 32 * XBW);
    float* xl = xm + 2 * 8 * GW;
    const uint32_t qt0 = smem_addr(smem + L.qt);  // the two query tiles, used by alternate units
    uint32_t qtbase = qt0;
    int uloc = 0;  // units of this CTA seen (the producer's count)
    const float scale = 1.4426950408889634f / sqrtf((float)D);
    // this lane's O^T rows are d = wg DW + 16 mt + 8 r + grp; bit 2 mt + r marks a probe
    // dim, pofs[2 mt + r] the byte offset of its slot in a record's partial rows
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
    const uint32_t part_base = smem_addr(smem + L.part);
    const int mi = lane >> 3, lr = lane & 7;
    const int keyK = wg * 16 + (mi & 1) * 8 + lr;  // K rows for the S^T A fragments
    const int chK = mi >> 1;
    const int keyV = (mi >> 1) * 8 + lr;  // V rows (within a 16-key chunk) for the O^T A fragments
    const int chV = mi & 1;
    const int PR = p.Ps < kBK ? p.Ps : kBK;
    const int lpr = 31 - __clz(PR);
    auto rowoff = [=](int row) -> uint32_t {
        return (uint32_t)(((row >> lpr) * (C::ROWB / 128) * PR + (row & (PR - 1))) * 128);
    };
    auto sw = [=](uint32_t base, int row, int chunk) -> uint32_t {
        return base + rowoff(row) + (uint32_t)((chunk >> 3) * PR * 128 + (((chunk & 7) ^ (row & 7)) << 4));
    };

    float acc[MT][4], tN[MT][4];
    float mrun[2], lrun[2], mbN[2], lbN[2];
    auto reset = [&]() {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mrun[j] = -INFINITY;
            lrun[j] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][c] = 0.f;
    };
    reset();
    mbN[0] = mbN[1] = lbN[0] = lbN[1] = 0.f;
    auto fold = [&]() {
        float a[2], bb[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const bool none = mbN[j] == -INFINITY;  // a head beyond G, or no valid key: keep the state
            const float mn = none ? mrun[j] : fmaxf(mrun[j], mbN[j]);
            a[j] = none ? 1.f : exp2f(mrun[j] - mn);
            bb[j] = none ? 0.f : exp2f(mbN[j] - mn);
            lrun[j] = none ? lrun[j] : a[j] * lrun[j] + bb[j] * lbN[j];
            mrun[j] = mn;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][c] = a[c & 1] * acc[mt][c] + bb[c & 1] * tN[mt][c];
    };
    int rec = 0;  // records published to the summary warp
    auto publish = [&](const UMeta& mt, int kind, bool data) -> bool {
        const int rb = rec % NB;
        if (rec >= NB && !wait_bounded(&part_empty[rb], (uint32_t)(rec / NB - 1) & 1u, ctrl, p.hdr, 242))
            return false;
        if (data) {
            // probe partial rows (high and low parts with the split tile); predicated stores
            const uint32_t rp = part_base + (uint32_t)(rb * C::PRW * C::PST * 4);
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const bool on = (pbits >> (2 * m + r)) & 1u;
                    if (G >= 2) st_shared_if(on && u1, rp + pofs[2 * m + r], tN[m][2 * r], tN[m][2 * r + 1]);
                    if (G % 2) st_shared_if(on && !u1, rp + pofs[2 * m + r], tN[m][2 * r]);
                }
            const bool lead = wg == 0 && grp == 0;
            st_shared_if(lead && w0, &plb[rb * G + (w0 ? q0 : 0)], lbN[0]);
            st_shared_if(lead && w1, &plb[rb * G + (w1 ? q1 : 0)], lbN[1]);
            st_shared_if(lead && w0, &pmb[rb * G + (w0 ? q0 : 0)], mbN[0]);
            st_shared_if(lead && w1, &pmb[rb * G + (w1 ? q1 : 0)], mbN[1]);
        }
        if (wg == 0 && lane == 0) {
            URec& r = rinfo[rb];
            r.kind = kind; r.item = mt.item; r.k = mt.k; r.j = mt.j; r.nj = mt.nj;
        }
        __syncwarp();
        mbar_arrive_if(lane == 0, &part_full[rb]);
        ++rec;
        return true;
    };
    // the unit's partial: this warp's dims of the [G][D] output sums; every warp holds
    // the same running max and weight sum, which warp 0 writes
    auto write_partial = [&](const UMeta& mt) {
        float* po;
        float* pml;
        if (mt.kind == kUFix) {
            const size_t ip = (size_t)mt.item * up.ck + mt.k;
            po = up.fix_o + ip * G * D;
            pml = up.fix_ml + ip * kUnitMlWords;
        } else {
            const size_t iu = (size_t)mt.item * up.maxk + mt.k;
            po = up.part_o + iu * G * D;
            pml = up.part_ml + iu * kUnitMlWords;
        }
        if constexpr (SPLITN) {
            // high + low parts (both lanes carry the same running max and sum)
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[m][c] += __shfl_xor_sync(0xffffffffu, acc[m][c], 2);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int d = wg * DW + 16 * m + 8 * r + grp;
                if (w0) po[q0 * D + d] = acc[m][2 * r];
                if (w1) po[q1 * D + d] = acc[m][2 * r + 1];
            }
        if (wg == 0 && grp == 0) {
            if (w0) {
                pml[q0] = mrun[0];
                pml[8 + q0] = lrun[0];
            }
            if (w1) {
                pml[q1] = mrun[1];
                pml[8 + q1] = lrun[1];
            }
        }
    };
    // bf16x2 multiplier 2^(e - emax) for a power-of-two exponent difference (0 below bf16 range)
    auto pow2_bf16x2 = [](float e, float emax) -> uint32_t {
        const float d = e - emax;  // an integer <= 0, or NaN / -inf
        const int k = d >= -126.f ? (int)d : -1000;
        const uint32_t bits = k >= -126 ? (uint32_t)(k + 127) << 7 : 0u;
        return bits | (bits << 16);
    };

    int xpar = 0;  // exchange buffer of the next block
    for (int e = 0;; ++e) {
        const int slot = e % p.stages;
        if (!wait_bounded(&full[slot], (uint32_t)(e / p.stages) & 1u, ctrl, p.hdr, 241)) return;
        const UMeta mt = meta[slot];
        const bool valid =
            mt.kind == kUEnd ||
            ((mt.kind == kUBlock || mt.kind == kUFix) && mt.item >= 0 && mt.item < p.num_items && mt.nvalid >= 1 &&
             mt.nvalid <= kBK && mt.nj >= 1 && mt.nj <= up.ck && mt.j >= 0 && mt.j < mt.nj && mt.k >= 0 &&
             mt.k < (mt.kind == kUFix ? up.ck : up.maxk) && mt.b >= 0 && mt.b < p.B && mt.g >= 0 && mt.g < p.Hkv);
        if (!valid || mt.kind == kUEnd) {
            if (!valid && lane == 0) record_check(p.hdr, 243, e, mt.kind, mt.item);
            __syncwarp();
            mbar_arrive_if(lane == 0, &empty[slot]);
            UMeta endm = mt;
            if (kART) publish(endm, kUEnd, false);
            return;
        }
        unsigned char* sK = ring + (size_t)slot * UC::SLOT;
        unsigned char* sV = sK + C::KVB;
        if (mt.j == 0) {
            // a new unit: its queries landed in tile uloc % 2 with this block
            reset();
            qtbase = qt0 + (uint32_t)((uloc & 1) * UC::QTB);
        }
        const int nvalid = mt.nvalid;
        // ---- S^T for this warp's 16 keys (two independent accumulation chains)
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
        const bool last = mt.j == mt.nj - 1;
        if (last) {
            // the unit's last read of its query tile: the producer may refill it
            __syncwarp();
            mbar_arrive_if(lane == 0, &qfree[uloc & 1]);
            ++uloc;
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
        // -inf / 0 for heads past G), then wait for the other warps
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
        named_bar_sync(1, GW * 32);
        // ---- the block's max exponent and weight sum per head
        {
            const float4 mq0 = *reinterpret_cast<const float4*>(xmp + (u0 ? q0 : 0) * GW);
            const float4 mq1 = *reinterpret_cast<const float4*>(xmp + (u1 ? q1 : 0) * GW);
            const float4 lq0 = *reinterpret_cast<const float4*>(xlp + (u0 ? q0 : 0) * GW);
            const float4 lq1 = *reinterpret_cast<const float4*>(xlp + (u1 ? q1 : 0) * GW);
            const float emx0 = fmaxf(fmaxf(mq0.x, mq0.y), fmaxf(mq0.z, mq0.w));
            const float emx1 = fmaxf(fmaxf(mq1.x, mq1.y), fmaxf(mq1.z, mq1.w));
            auto wsum = [](const float4& m, const float4& l, float mx) {
                float s = 0.f;
                s += m.x == -INFINITY ? 0.f : exp2f(m.x - mx) * l.x;
                s += m.y == -INFINITY ? 0.f : exp2f(m.y - mx) * l.y;
                s += m.z == -INFINITY ? 0.f : exp2f(m.z - mx) * l.z;
                s += m.w == -INFINITY ? 0.f : exp2f(m.w - mx) * l.w;
                return s;
            };
            mbN[0] = u0 ? emx0 : -INFINITY;
            mbN[1] = u1 ? emx1 : -INFINITY;
            lbN[0] = u0 && emx0 != -INFINITY ? wsum(mq0, lq0, emx0) : 0.f;
            lbN[1] = u1 && emx1 != -INFINITY ? wsum(mq1, lq1, emx1) : 0.f;
        }
        const float4 mb4 = *reinterpret_cast<const float4*>(xmp + hb * GW);
        const float ebh = fmaxf(fmaxf(mb4.x, mb4.y), fmaxf(mb4.z, mb4.w));
        const float mbw[4] = {mb4.x, mb4.y, mb4.z, mb4.w};
        // ---- O^T of this warp's dims over the block's 64 keys, chunk by chunk, in two
        // independent accumulator chains (even chunks or high parts into tN, odd chunks or
        // low parts into tN2) that are added at the end
        float tN2[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            tN[m][0] = tN[m][1] = tN[m][2] = tN[m][3] = 0.f;
            tN2[m][0] = tN2[m][1] = tN2[m][2] = tN2[m][3] = 0.f;
        }
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
                if constexpr (SPLITN) {
                    mma_bf16((c & 1) ? tN2[m] : tN[m], a0, a1, a2, a3, b[0], b[1]);
                } else {
                    mma_bf16(tN[m], a0, a1, a2, a3, b[0], b[1]);
                    mma_bf16(tN2[m], a0, a1, a2, a3, b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int c = 0; c < 4; ++c) tN[m][c] += tN2[m][c];
        xpar ^= 1;
        __syncwarp();
        mbar_arrive_if(lane == 0, &empty[slot]);  // the slot's data are no longer read
        if (kART && mt.kind == kUBlock && !publish(mt, kUBlock, true)) return;
        fold();
        if (last) write_partial(mt);
    }
}

// ---------------------------------------------------------------------------
// helpers of the two statistics roles
// ---------------------------------------------------------------------------
// (M1, L1, O1) <- merge with (M2, L2, O2): the same softmax state over both sets of blocks
template <int SPL>
__device__ __forceinline__ void state_merge(float& M1, float& L1, float (&O1)[SPL], float M2, float L2,
                                            const float (&O2)[SPL]) {
    if (M2 == -INFINITY) return;
    const float Mn = fmaxf(M1, M2);
    const float a = exp2f(M1 - Mn), bw = exp2f(M2 - Mn);
    L1 = fmaf(a, L1, bw * L2);
#pragma unroll
    for (int j = 0; j < SPL; ++j) O1[j] = fmaf(a, O1[j], bw * O2[j]);
    M1 = Mn;
}

// Probe slot s = lane + 32 j is word s of a partial row: head s % GP, rank s / GP; hs[j] is
// its head, or -1 past the probe (heads from p.ph on are not part of it). All slots of a
// lane belong to head hme.
template <class C>
__device__ __forceinline__ void probe_slots(const Params& p, int lane, int (&hs)[C::SPL], int& hme) {
#pragma unroll
    for (int j = 0; j < C::SPL; ++j) {
        const int s = lane + 32 * j;
        hs[j] = (s % C::GP < p.ph && s / C::GP < p.m) ? s % C::GP : -1;
    }
    hme = lane % C::GP < C::GQ ? lane % C::GP : 0;
}

// ---------------------------------------------------------------------------
// summary warp: the consumers' block records become block summaries in the
// unit store; at a unit's end it publishes the unit's probe aggregate and hands
// the unit to the test warp
// ---------------------------------------------------------------------------
template <class C>
__device__ void summ_u(const Params& p, const UParams& up, const float* part, const float* plb, const float* pmb,
                       uint64_t* part_full, uint64_t* part_empty, const URec* rinfo, float* ust, URec* uhdr,
                       uint64_t* ufull, uint64_t* uempty, uint64_t* ustart, Ctrl* ctrl) {
    constexpr int G = C::GQ, SPL = C::SPL, RGW = C::RGW, W = SPL + 2;
    constexpr int UBUF = kUnitBlocks * kUnitWords * 32;  // floats of one summary buffer
    constexpr int NPR = C::RGW * C::PRW;  // partial rows per record
    constexpr int UW = 32 * kUnitWords;   // floats of one probe state in the workspace
    const int lane = threadIdx.x & 31;
    int hs[SPL], hme;
    probe_slots<C>(p, lane, hs, hme);
    float Ma = -INFINITY, La = 0.f, Oa[SPL];  // aggregate of the current unit's blocks
#pragma unroll
    for (int j = 0; j < SPL; ++j) Oa[j] = 0.f;
    int urec = 0;  // units handed to the test warp
    for (int rec = 0;; ++rec) {
        const int rb = rec % kUnitRecs;
        if (!wait_bounded(&part_full[rb], (uint32_t)(rec / kUnitRecs) & 1u, ctrl, p.hdr, 251)) return;
        const URec ri = rinfo[rb];
        const bool valid = ri.kind == kUBlock && ri.j >= 0 && ri.j < ri.nj && ri.nj <= up.ck && ri.item >= 0 &&
                           ri.item < p.num_items && ri.k >= 0 && ri.k < up.maxk;
        // a new unit (or the end) needs its summary buffer (urec % 2) back from the test
        // warp, which released it after the tests of the unit two before
        const int ub = urec & 1;
        if ((!valid || ri.j == 0) && urec >= 2 &&
            !wait_bounded(&uempty[ub], (uint32_t)((urec >> 1) - 1) & 1u, ctrl, p.hdr, 255))
            return;
        if (!valid) {
            if (ri.kind == kUBlock && lane == 0) record_check(p.hdr, 254, ri.item, ri.k, ri.j);
            URec e = ri;
            e.kind = kUEnd;
            if (lane == 0) {
                uhdr[ub] = e;
                uhdr[2 + ub] = e;
            }
            __syncwarp();
            mbar_arrive_if(lane == 0, &ufull[ub]);
            mbar_arrive_if(lane == 0, &ustart[ub]);
            return;
        }
        if (ri.j == 0) {
            // the test warp may start the unit's look-back while its blocks are computed
            if (lane == 0) uhdr[2 + ub] = ri;
            __syncwarp();
            mbar_arrive_if(lane == 0, &ustart[ub]);
        }
        // block max and weight sum of this lane's head over the 4 warps (each used its own
        // max), and the block's probe sums at that max
        float sw[RGW];
        float mbk = -INFINITY;
#pragma unroll
        for (int w = 0; w < RGW; ++w) {
            sw[w] = pmb[(rb * RGW + w) * G + hme];
            mbk = fmaxf(mbk, sw[w]);
        }
        float lb = 0.f;
#pragma unroll
        for (int w = 0; w < RGW; ++w) {
            sw[w] = sw[w] == -INFINITY ? 0.f : exp2f(sw[w] - mbk);  // a warp without valid keys adds nothing
            lb = fmaf(sw[w], plb[(rb * RGW + w) * G + hme], lb);
        }
        const float* pp = part + (size_t)rb * NPR * C::PST;
        float pb[SPL];
#pragma unroll
        for (int j = 0; j < SPL; ++j) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < RGW; ++w) {
                float pw = 0.f;
#pragma unroll
                for (int r = 0; r < C::PRW; ++r) pw += pp[(w * C::PRW + r) * C::PST + lane + 32 * j];
                v = fmaf(sw[w], pw, v);
            }
            pb[j] = hs[j] >= 0 ? v : 0.f;  // slots past the probe hold no data
        }
        __syncwarp();
        mbar_arrive_if(lane == 0, &part_empty[rb]);
        float* sm = ust + (size_t)ub * UBUF + (size_t)ri.j * W * 32;
        sm[lane] = mbk;
        sm[32 + lane] = lb;
#pragma unroll
        for (int j = 0; j < SPL; ++j) sm[(2 + j) * 32 + lane] = pb[j];
        if (ri.j == 0) {
            Ma = mbk;
            La = lb;
#pragma unroll
            for (int j = 0; j < SPL; ++j) Oa[j] = pb[j];
        } else {
            state_merge<SPL>(Ma, La, Oa, mbk, lb, pb);
        }
        if (ri.j == ri.nj - 1) {
            // the unit's aggregate for the look-backs of later units, and for the test warp
            const size_t iu = (size_t)ri.item * up.maxk + ri.k;
            float* ga = up.agg + iu * UW;
            ga[lane] = Ma;
            ga[32 + lane] = La;
#pragma unroll
            for (int j = 0; j < SPL; ++j) ga[(2 + j) * 32 + lane] = Oa[j];
            if (lane == 0) uhdr[ub] = ri;
            __syncwarp();
            mbar_arrive_if(lane == 0, &ufull[ub]);  // the summaries and the aggregate are written
            ++urec;
            fence_acq_rel_gpu();
            __syncwarp();
            if (lane == 0) st_release_gpu(&up.tflag[iu], 1);
        }
    }
}

// ---------------------------------------------------------------------------
// test warp: per unit handed over by the summary warp, the look-back for the
// probe state before the unit, the stability tests of its blocks, and its stop
// ---------------------------------------------------------------------------
template <class C>
__device__ void stat_u(const Params& p, const UParams& up, const float* ust, const URec* uhdr, uint64_t* ufull,
                       uint64_t* uempty, uint64_t* ustart, Ctrl* ctrl) {
    constexpr int UBUF = kUnitBlocks * kUnitWords * 32;  // floats of one summary buffer
    bool released = false;  // the unit's summary buffer has been handed back to the summary warp
    int ub = 0;             // ... which of the two
    auto release_buffer = [&]() {
        if (released) return;
        __syncwarp();
        mbar_arrive_if((threadIdx.x & 31) == 0, &uempty[ub]);
        released = true;
    };
    constexpr int SPL = C::SPL;
    constexpr int W = SPL + 2;
    constexpr int UW = 32 * kUnitWords;  // floats of one probe state in the workspace
    const int lane = threadIdx.x & 31;
    int hs[SPL], hme;
    probe_slots<C>(p, lane, hs, hme);
    (void)hme;

    // the probe state before unit k of the item: aggregates of the earlier units, back to
    // the nearest one with an inclusive state (dead: a unit before it was skipped, so the
    // item stopped before it). Taken when the unit starts, while its blocks are computed.
    auto lookback = [&](int item, int k, float& cM, float& cL, float (&cO)[SPL], bool& dead) -> bool {
        cM = -INFINITY;
        cL = 0.f;
#pragma unroll
        for (int j = 0; j < SPL; ++j) cO[j] = 0.f;
        dead = false;
        {
            // lane j reads the flag of unit kk - j; the lanes from 0 up to the first unit with an
            // inclusive state (or a skip mark, or the list's start) whose states are published
            // are folded together, their loads in flight at once
            const size_t ibase = (size_t)item * up.maxk;
            const unsigned long long t0 = global_ns();
            int kk = k - 1;
            for (unsigned it = 0; kk >= 0; ++it) {
                const int uj = kk - lane;
                const int fl = uj >= 0 ? ld_acquire_gpu(&up.tflag[ibase + uj]) : 2;  // before the list: empty
                const unsigned pub = __ballot_sync(0xffffffffu, fl >= 1);
                const unsigned endm = __ballot_sync(0xffffffffu, fl >= 2);
                const int r = pub == 0xffffffffu ? 32 : __ffs(~pub) - 1;  // lanes 0 .. r-1 published
                const int e = endm ? __ffs(endm) - 1 : 32;                // first inclusive / skipped / start
                if (r == 0) {
                    int quit = 0;
                    if (lane == 0) {
                        if (ld_volatile_shared(&ctrl->abort)) quit = 1;
                        else if ((it & 63u) == 63u && global_ns() - t0 > ctrl->wait_ns) {
                            st_volatile_shared(&ctrl->abort, 1);
                            atomicOr(&p.hdr->status, ART_STATUS_TIMEOUT);
                            record_check(p.hdr, 252, item, kk, k);
                            quit = 1;
                        }
                    }
                    if (__shfl_sync(0xffffffffu, quit, 0)) return false;
                    __nanosleep(64);
                    continue;
                }
                const int take = e < r ? e + 1 : r;
                if (e < take && __shfl_sync(0xffffffffu, fl, e) == 3) {
                    dead = true;  // a unit before this one was skipped: the item stopped before it
                    break;
                }
                for (int t = 0; t < take; t += 4) {
                    float M2[4], L2[4], O2[4][SPL];
                    int ft[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int tq = t + q;
                        const int ut = kk - tq;
                        const int f = __shfl_sync(0xffffffffu, fl, tq & 31);
                        ft[q] = (tq < take && ut >= 0) ? f : 0;
                        // every lane orders its payload loads after its own acquire of the flag
                        if (ft[q]) (void)ld_acquire_gpu(&up.tflag[ibase + ut]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int ut = max(kk - (t + q), 0);
                        const float* src = (ft[q] == 2 ? up.incl : up.agg) + (ibase + ut) * UW;
                        M2[q] = ft[q] ? __ldcg(src + lane) : -INFINITY;
                        L2[q] = ft[q] ? __ldcg(src + 32 + lane) : 0.f;
#pragma unroll
                        for (int j = 0; j < SPL; ++j) O2[q][j] = ft[q] ? __ldcg(src + (2 + j) * 32 + lane) : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) state_merge<SPL>(cM, cL, cO, M2[q], L2[q], O2[q]);
                }
                if (e < take) break;  // reached an inclusive state or the list's start
                kk -= take;
            }
        }
        return true;
    };

    // until every block of buffer ub's unit (item, k) is summarized and its aggregate written
    auto wait_unit = [&](int uu, int item, int k) -> bool {
        if (!wait_bounded(&ufull[ub], (uint32_t)(uu >> 1) & 1u, ctrl, p.hdr, 251)) return false;
        const URec ri = uhdr[ub];
        if (ri.kind != kUBlock || ri.item != item || ri.k != k) {
            if (lane == 0) record_check(p.hdr, 257, ri.item, ri.k, k);
            return false;
        }
        return true;
    };

    auto finish_unit = [&](int uu, int item, int k, int nj, float cM, float cL, const float (&cO)[SPL],
                           bool dead) -> bool {
        const size_t iu = (size_t)item * up.maxk + k;
        const float* us = ust + (size_t)ub * UBUF;
        int* uf = up.uflags + 4 * iu;
        if (dead) {
            if (!wait_unit(uu, item, k)) return false;
            if (lane == 0) {
                st_release_gpu(&up.tflag[iu], 3);
                st_release_gpu(uf + 2, 3);
            }
        } else {
            if (!wait_unit(uu, item, k)) return false;
            {
                // the unit's own aggregate, written by the summary warp before it handed the
                // unit over, and the inclusive state (its flag follows after the first pass)
                float Ma, La, Oa[SPL];
                const float* ga = up.agg + iu * UW;
                Ma = ga[lane];
                La = ga[32 + lane];
#pragma unroll
                for (int j = 0; j < SPL; ++j) Oa[j] = ga[(2 + j) * 32 + lane];
                float iM = cM, iL = cL, iO[SPL];
#pragma unroll
                for (int j = 0; j < SPL; ++j) iO[j] = cO[j];
                state_merge<SPL>(iM, iL, iO, Ma, La, Oa);
                float* gi = up.incl + iu * UW;
                gi[lane] = iM;
                gi[32 + lane] = iL;
#pragma unroll
                for (int j = 0; j < SPL; ++j) gi[(2 + j) * 32 + lane] = iO[j];
            }
            // the stability test of each block of the unit, in list order, from that state
            float M = cM, Lsum = cL, X[SPL];
            const float rL = cL > 0.f ? 1.f / cL : 0.f;
            float q = 0.f;
#pragma unroll
            for (int j = 0; j < SPL; ++j) {
                X[j] = hs[j] >= 0 ? cO[j] * rL : 0.f;
                q = fmaf(X[j], X[j], q);
            }
            q = warp_sum(q);
            const float n0 = sqrtf(q);  // |x| before the unit's first block
            // pass 1, lane-local: the probe's change over each block (the update of x is
            // per slot), and this lane's terms of sum delta^2, sum delta . x_{i-1}, |x_i|^2
            constexpr int VS = 16;  // entries per statistic (>= kUnitBlocks; 4 VS a power of two)
            static_assert(VS >= kUnitBlocks, "one entry per block");
            float v[4 * VS];
#pragma unroll
            for (int j = 0; j < 4 * VS; ++j) v[j] = 0.f;
            // the summaries (in global memory) are read four blocks at a time, with the
            // loads of the four in flight together
            constexpr int BQ = 4;
            static_assert(kUnitBlocks % BQ == 0, "whole batches");
#pragma unroll
            for (int j0 = 0; j0 < kUnitBlocks; j0 += BQ) {
                float sv[BQ][W];
#pragma unroll
                for (int q = 0; q < BQ; ++q) {
                    const float* s = us + (size_t)(j0 + q) * W * 32;
                    const bool live = j0 + q < nj;
#pragma unroll
                    for (int x = 0; x < W; ++x) sv[q][x] = live ? s[x * 32 + lane] : 0.f;
                }
#pragma unroll
                for (int q = 0; q < BQ; ++q) {
                    const int j = j0 + q;
                    float s1 = 0.f, s2 = 0.f, s3 = 0.f;
                    if (j < nj) {
                        const float mbk = sv[q][0], lb = sv[q][1];
                        const float Mn = fmaxf(M, mbk);
                        const float a = exp2f(M - Mn);
                        const float bw = exp2f(mbk - Mn);
                        const float Ln = fmaf(a, Lsum, bw * lb);
                        const float cf = __fdividef(bw, Ln);
                        M = Mn;
                        Lsum = Ln;
#pragma unroll
                        for (int jj = 0; jj < SPL; ++jj) {
                            const float pb = sv[q][2 + jj];
                            const float d = hs[jj] >= 0 ? cf * (pb - lb * X[jj]) : 0.f;
                            s1 = fmaf(d, d, s1);
                            s2 = fmaf(d, X[jj], s2);
                            X[jj] += d;
                            s3 = fmaf(X[jj], X[jj], s3);
                        }
                    }
                    v[j] = s1;
                    v[VS + j] = s2;
                    v[2 * VS + j] = s3;
                }
            }
            release_buffer();  // the summaries are read: the summary warp may fill in the next unit's
            fence_acq_rel_gpu();
            __syncwarp();
            if (lane == 0) st_release_gpu(&up.tflag[iu], 2);  // the inclusive state
            // pass 2: the warp sums of all of them at once; lane l then holds the sums of
            // entries 2 l and 2 l + 1
            transpose_reduce<4 * VS, 32>(v, lane);
            auto sum_at = [&](int entry) -> float {  // warp sum of entry `entry`, in every lane
                const float a0 = __shfl_sync(0xffffffffu, v[0], (entry >> 1) & 31);
                const float a1 = __shfl_sync(0xffffffffu, v[1], (entry >> 1) & 31);
                return (entry & 1) ? a1 : a0;
            };
            // pass 3: lane b takes the test of block b, the same tests as the one-CTA
            // statistics warp, multiplied through by their positive denominators
            const int bj = lane < kUnitBlocks ? lane : 0;
            const float s1 = sum_at(bj), s2 = sum_at(VS + bj), s3 = sum_at(2 * VS + bj);
            const float s3p = sum_at(2 * VS + (bj > 0 ? bj - 1 : 0));
            const float nprev = bj == 0 ? n0 : sqrtf(s3p);
            const float rprev = bj == 0 ? (n0 > 0.f ? 1.f / n0 : 0.f) : __fdividef(1.f, nprev);
            const float ni = sqrtf(s3);
            const float S = ni + nprev, T = 2.f * s2 + s1;
            const bool mag_ok = fabsf(T) * rprev < p.eps_mag * S;
            const float Nd = fmaf(s1, S * S, fmaf(-2.f * s2 * T, S * rprev, T * T));
            const bool dir_ok = fmaxf(0.f, Nd) < 2.f * p.eps_dir * s3 * (S * S);
            const int pos = k * up.ck + bj;
            const bool stable = lane < nj && pos >= 1 && nprev > 0.f && ni > 0.f && nprev < 1e30f && ni < 1e30f &&
                                mag_ok && dir_ok;
            const uint32_t bits = __ballot_sync(0xffffffffu, stable);
            if (lane == 0) {
                uf[0] = (int)bits;
                uf[1] = nj;
                st_release_gpu(uf + 2, 1);
            }
            // the patience count entering the unit: the previous unit's trailing stable run
            int counter = 0;
            bool dead2 = false;
            if (k > 0) {
                const int* pf = up.uflags + 4 * (iu - 1);
                int st = 0;
                if (!poll_flag(pf + 2, 1, st, ctrl, p.hdr, 253)) return false;
                if (st == 3) {
                    dead2 = true;
                } else {
                    const uint32_t pbits = (uint32_t)__ldcg(pf);
                    const int pn = __ldcg(pf + 1);
                    int run = 0;
                    for (int jj = pn - 1; jj >= 0 && ((pbits >> jj) & 1u); --jj) ++run;
                    counter = min(run, p.patience);
                }
            }
            if (!dead2) {
                const ItemInfo inf = p.info[item];
                const int n = inf.n;
                const bool has0 = (inf.flags & kItemHas0) != 0;
                const int pz = up.p0[item];
                int cand = -1;
                for (int j = 0; j < nj; ++j) {
                    const int pos = k * up.ck + j;
                    const bool st = (bits >> j) & 1u;
                    counter = st ? min(counter + 1, p.patience) : 0;
                    const bool seen0 = !has0 || pos >= pz;
                    if (pos == n - 1 || (st && counter >= p.patience && seen0)) {
                        cand = pos;
                        break;
                    }
                }
                if (cand >= 0 && lane == 0) atomicMin(&up.stop_min[item], cand);
            }
        }
        __syncwarp();
        if (lane == 0) {
            st_release_gpu(up.uflags + 4 * iu + 3, 1);  // resolved: after this lane's atomicMin and flags
            red_release_add(&up.resolved[item], 1);
        }
        return true;
    };

    for (int uu = 0;; ++uu) {
        ub = uu & 1;
        // the unit that started in buffer ub: its look-back, then (once its blocks are
        // summarized) its tests
        if (!wait_bounded(&ustart[ub], (uint32_t)(uu >> 1) & 1u, ctrl, p.hdr, 256)) return;
        const URec rs = uhdr[2 + ub];
        if (rs.kind != kUBlock) return;
        released = false;
        float cM, cL, cO[SPL];
        bool dead;
        if (!lookback(rs.item, rs.k, cM, cL, cO, dead)) return;
        const bool done = finish_unit(uu, rs.item, rs.k, rs.nj, cM, cL, cO, dead);
        release_buffer();  // a unit whose item had stopped before it has not read its summaries
        if (!done) return;
    }
}

// ---------------------------------------------------------------------------
// the kernels
// ---------------------------------------------------------------------------
template <int D, int G, bool kART>
__global__ void __launch_bounds__(UCfg<D, G>::THREADS, 2)
    art_units_kernel(const Params p, const UParams up0, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tq) {
    UParams up = up0;
    up.ck = p.hdr->ck;  // chosen by the plan kernel
    using C = typename UCfg<D, G>::C;
    using UC = UCfg<D, G>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const ULayout L = make_ulayout<D, G>(p.stages);
    unsigned char* ring = smem;
    UMeta* meta = reinterpret_cast<UMeta*>(smem + L.meta);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + p.stages;
    uint64_t* part_full = empty + p.stages;
    uint64_t* part_empty = part_full + kUnitRecs;
    uint64_t* ufull = part_empty + kUnitRecs;  // [2]
    uint64_t* uempty = ufull + 2;              // [2]
    uint64_t* stall_bar = uempty + 2;  // never completed (the failure-path test hook)
    uint64_t* qfree = stall_bar + 1;    // [2]: the consumers are done with a query tile
    uint64_t* ustart = qfree + 2;       // [2]: a unit has started in summary buffer 0 / 1
    float* ust = up.ustore + (size_t)blockIdx.x * 2 * kUnitBlocks * kUnitWords * 32;  // this CTA's summary store
    int* prank = reinterpret_cast<int*>(smem + L.ptab);
    URec* rinfo = reinterpret_cast<URec*>(smem + L.rinfo);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + L.ctrl);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::GW);
        }
        for (int b = 0; b < kUnitRecs; ++b) {
            mbar_init(&part_full[b], C::GW);
            mbar_init(&part_empty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ufull[b], 1);
            mbar_init(&uempty[b], 1);
        }
        mbar_init(stall_bar, 1);
        mbar_init(&qfree[0], C::GW);
        mbar_init(&qfree[1], C::GW);
        mbar_init(&ustart[0], 1);
        mbar_init(&ustart[1], 1);
        ctrl->stop_item = -1;
        ctrl->abort = 0;
        ctrl->wait_ns = p.wait_ns;
        fence_mbar_init();
    }
    if (tid < D) {
        // rank of head dim `tid` among the probe dims, or -1
        int found = 0, rank = 0;
        for (int k = 0; k < p.m; ++k) {
            const int col = p.probe[k];
            if (col == tid) found = 1;
            if (col >= 0 && col < tid) ++rank;
        }
        prank[tid] = found ? rank : -1;
    }
    if (tid == 4 * 32) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tv)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tq)) : "memory");
    }
    __syncthreads();
    const int warp = tid >> 5;
    if (p.stall && warp < 4 && !wait_bounded(stall_bar, 0u, ctrl, p.hdr, 261 + 1)) return;
    if (warp == 4) {
        producer_u<C, UC>(p, up, ring, meta, full, empty, qfree, smem + L.qt, ctrl, &tk, &tv, &tq);
    } else if (warp == 5) {
        if (kART)
            summ_u<C>(p, up, reinterpret_cast<const float*>(smem + L.part), reinterpret_cast<const float*>(smem + L.plb),
                      reinterpret_cast<const float*>(smem + L.pmb), part_full, part_empty, rinfo,
                      ust, reinterpret_cast<URec*>(smem + L.uhdr), ufull, uempty, ustart, ctrl);
    } else if (warp == 6) {
        if (kART)
            stat_u<C>(p, up, ust, reinterpret_cast<const URec*>(smem + L.uhdr), ufull, uempty, ustart, ctrl);
    } else {
        consumer_u<C, UC, kART>(p, up, ring, meta, full, empty, part_full, part_empty, qfree, rinfo, L, smem, prank,
                                ctrl);
    }
}

// Per (item, query head): merge the partials of the units before the stopping unit and
// of the fix pieces (or of the stopping unit itself when it ends at the stop), and write
// O = sums / weight sums and blocks_used. The CTA's kCombineSplit x D threads first load
// every partial's max and weight sum together (one partial per thread), reduce them to
// the common max and the weight sum, and turn the maxima into factors; then thread
// (s, d) adds head dim d's weighted sums of partials s, s + kCombineSplit, ..., all its
// loads in flight at once, and the kCombineSplit sums of a dim are added in a fixed
// order (reproducible results).
constexpr int kCombineSplit = 4;                      // threads per head dim
constexpr int kCombineInFlight = 16;                  // loads of one thread in flight

template <int D, int G>
__global__ void __launch_bounds__(D * kCombineSplit) art_units_combine(const Params p, const UParams up0) {
    using E = Elem<true>;
    constexpr int NT = D * kCombineSplit, NW = NT / 32;
    // launched while the unit kernel may still run: wait for it to finish
    asm volatile("griddepcontrol.wait;" ::: "memory");
    UParams up = up0;
    up.ck = p.hdr->ck;
    extern __shared__ float s_dyn[];
    float* s_f = s_dyn;                          // [maxk + kUnitBlocks] the partials' maxima, then factors
    float* s_l = s_dyn + up0.maxk + kUnitBlocks;  // [maxk + kUnitBlocks] the partials' weight sums
    __shared__ float s_red[2][NW];
    __shared__ float s_sum[kCombineSplit][D];
    const int item = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int d = tid % D, sp = tid / D;
    const int lane = tid & 31, wq = tid >> 5;
    const bool lead = tid == 0 && h == 0;
    const int b = item / p.Hkv, g = item - (item / p.Hkv) * p.Hkv;
    const size_t obase = ((size_t)b * p.Hq + (size_t)g * G + h) * D;
    const ItemInfo inf = p.info[item];
    const bool bad = (inf.flags & kItemBad) || up.fail[item] != 0;
    const int n = bad ? 0 : inf.n;
    const int t = n > 0 ? up.stop_min[item] : -1;
    if (bad || n == 0 || t < 0 || t >= n) {
        if (!bad && n > 0 && lead) record_check(p.hdr, 261, item, t, n);
        if (sp == 0) E::store(p.out, obase + d, 0.f);
        if (lead && p.blocks_used) p.blocks_used[item] = (bad || n > 0) ? -1 : 0;
        return;
    }
    if (lead && p.blocks_used) p.blocks_used[item] = t + 1;
    const int kk = t / up.ck, sfirst = kk * up.ck;
    const bool use_fix = t != min(n, sfirst + up.ck) - 1;
    const int nunits = use_fix ? kk : kk + 1;                // whole units
    const int nq = nunits + (use_fix ? t - sfirst + 1 : 0);  // ... then fix pieces (one block each)
    if (nq > up.maxk + kUnitBlocks) {  // beyond the workspace's sizing: cannot happen for a checked plan
        if (lead) record_check(p.hdr, 263, item, nq, up.maxk + kUnitBlocks);
        return;
    }
    const size_t ubase = (size_t)item * up.maxk, fbase = (size_t)item * up.ck - nunits;
    auto ml_of = [&](int q) -> const float* {
        return q < nunits ? up.part_ml + (ubase + q) * kUnitMlWords : up.fix_ml + (fbase + q) * kUnitMlWords;
    };
    auto o_of = [&](int q) -> const float* {
        return q < nunits ? up.part_o + (ubase + q) * G * D : up.fix_o + (fbase + q) * G * D;
    };
    // the common max (the weight sums are loaded with the maxima)
    float mx = -INFINITY;
    for (int q = tid; q < nq; q += NT) {
        const float* ml = ml_of(q);
        const float m = __ldcg(ml + h);
        s_l[q] = __ldcg(ml + 8 + h);
        s_f[q] = m;
        mx = fmaxf(mx, m);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[0][wq] = mx;
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_red[0][w]);
    // factors and the weight sum
    float den = 0.f;
    for (int q = tid; q < nq; q += NT) {
        const float m = s_f[q];
        const float f = m == -INFINITY ? 0.f : exp2f(m - M);
        s_f[q] = f;
        den = fmaf(f, s_l[q], den);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane == 0) s_red[1][wq] = den;
    __syncthreads();
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) L += s_red[1][w];
    // this thread's share of dim d's weighted sums: partials sp, sp + kCombineSplit, ...
    float num = 0.f;
    for (int q0 = sp; q0 < nq; q0 += kCombineSplit * kCombineInFlight) {
        float v[kCombineInFlight];
#pragma unroll
        for (int x = 0; x < kCombineInFlight; ++x) {
            const int q = q0 + x * kCombineSplit;
            v[x] = q < nq ? __ldcg(o_of(q) + h * D + d) : 0.f;
        }
#pragma unroll
        for (int x = 0; x < kCombineInFlight; ++x) {
            const int q = q0 + x * kCombineSplit;
            if (q < nq) num = fmaf(s_f[q], v[x], num);
        }
    }
    s_sum[sp][d] = num;
    __syncthreads();
    if (sp == 0) {
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < kCombineSplit; ++k) tot += s_sum[k][d];
        E::store(p.out, obase + d, tot / L);
    }
}

// Largest ring depth (2..8 slots) that lets `want` CTAs share one SM.
template <int D, int G>
inline int pick_ustages(int want, int smem_per_sm, int smem_per_block) {
    for (int s = 8; s >= 2; --s) {
        const size_t t = make_ulayout<D, G>(s).total;
        if ((int)t <= smem_per_block && (size_t)want * (t + 1024) <= (size_t)smem_per_sm) return s;
    }
    return 0;
}

template <int D, int G, bool kART>
cudaError_t launch_units(Params p, UParams up, cudaStream_t stream, LaunchInfo* li) {
    auto kern = art_units_kernel<D, G, kART>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 0, smem_sm = 0, smem_blk = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    const char* envs = std::getenv("ART_STAGES");
    const int force = envs ? std::atoi(envs) : 0;
    int stages = force >= 2 && force <= 8 ? force : pick_ustages<D, G>(2, smem_sm, smem_blk);
    if (stages == 0) stages = pick_ustages<D, G>(1, smem_sm, smem_blk);
    if (stages == 0) return cudaErrorInvalidConfiguration;
    const size_t smem = make_ulayout<D, G>(stages).total;
    if ((int)smem > smem_blk) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    int occ = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, UCfg<D, G>::THREADS, smem)) != cudaSuccess)
        return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof tk);
    std::memset(&tv, 0, sizeof tv);
    const long long rows = (long long)p.num_pages * p.Hkv * p.Ps;
    if (rows >= (1LL << 31)) return cudaErrorInvalidValue;
    const char* env3 = std::getenv("ART_TMA3D");
    p.tma3d = (!env3 || std::atoi(env3) != 0) && make_cache_map3(&tk, p.k, rows, D, p.Ps) == cudaSuccess &&
              make_cache_map3(&tv, p.v, rows, D, p.Ps) == cudaSuccess;
    if (!p.tma3d) {
        if ((e = make_cache_map(&tk, p.k, rows, D, p.Ps)) != cudaSuccess) return e;
        if ((e = make_cache_map(&tv, p.v, rows, D, p.Ps)) != cudaSuccess) return e;
    }
    // the queries [batch * Hq rows][D], read 8 rows (one group's heads and the next's) at a time
    CUtensorMap tq;
    std::memset(&tq, 0, sizeof tq);
    const long long qrows = (long long)p.B * p.Hq;
    if (p.tma3d) {
        if ((e = make_cache_map3(&tq, p.q, qrows, D, 8)) != cudaSuccess) return e;
    } else {
        if ((e = make_cache_map(&tq, p.q, qrows, D, 8)) != cudaSuccess) return e;
    }
    p.stages = stages;
    const int grid = sms * occ < kUnitMaxCtas ? sms * occ : kUnitMaxCtas;
    if (li) {
        li->grid = grid;
        li->stages = stages;
        li->smem = smem;
        li->ctas_per_sm = occ;
    }
    kern<<<grid, UCfg<D, G>::THREADS, smem, stream>>>(p, up, tk, tv, tq);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the merge kernel may start while the unit kernel drains (programmatic dependent
    // launch); it waits for the unit kernel's completion before reading anything
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(p.num_items, G, 1);
    cfg.blockDim = dim3(D * kCombineSplit);
    // the partials' maxima and weight sums: up to maxk units and kUnitBlocks fix pieces
    cfg.dynamicSmemBytes = (size_t)2 * (up.maxk + kUnitBlocks) * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, art_units_combine<D, G>, p, up);
}

}  // namespace art

#define ART_UNITS_INSTANTIATE(D, G)                                                                      \
    template cudaError_t art::launch_units<D, G, true>(art::Params, art::UParams, cudaStream_t,           \
                                                       art::LaunchInfo*);                                 \
    template cudaError_t art::launch_units<D, G, false>(art::Params, art::UParams, cudaStream_t,          \
                                                        art::LaunchInfo*);
