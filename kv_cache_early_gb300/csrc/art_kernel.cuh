// art_kernel.cuh -- the persistent, warp-specialized ART decode-attention kernel.
//
// One CTA runs three roles over a ring of `stages` shared-memory slots, each
// slot holding one 64-token ART block of K rows, V rows and (for an item's
// first block) the item's G query vectors:
//
//   producer warp   claims work items (sequence b, KV head g) in the order the
//                   plan kernel wrote (longest visit list first), resolves
//                   visit entry -> logical block -> physical pages through the
//                   block table, and fills slots with cp.async.bulk copies that
//                   complete on the slot's mbarrier. It stops issuing an item's
//                   blocks once the statistics warp has stopped that item.
//   consumer warps  (kNWC) each own 8 of the block's 64 rows. Scores
//                   s = q.k * log2(e)/sqrt(d) in fp32; the block's largest
//                   score per head is shared through a named barrier; weights
//                   p = 2^(s - m_blk); the block's P.V partial; and an online-
//                   softmax fold into the running accumulators (ART paper
//                   sec. 3.1: FlashAttention's streaming softmax, O^(t) after
//                   t blocks). Arithmetic on packed fp32 pairs (f32x2).
//   statistics warp merges the consumer warps' block sums and P.V at the probe
//                   columns, in visit order, into the probe x^(i) of O^(i), and
//                   evaluates the stability test (magnitude and direction
//                   change both below their thresholds for `patience`
//                   consecutive blocks, never before block 0 has been
//                   processed) -- ART paper sec. 3.2, gist.science explainer
//                   sec. 2.2-2.4.
//
// The consumers do not wait for the decision on block i before computing
// block i+1 (G <= 4): block i+1 is held apart and folded only once block i's
// decision says "continue"; after a stop it is discarded. For G > 4 (register
// budget) each block waits for its own decision.
//
// The statistics avoid cancellation: the change of the probe over block i is
// formed directly, delta = b (P.V_probe - l_blk x^(i-1)) / L_i, the norm
// change as delta.(2x + delta) / (|x_i| + |x_{i-1}|), and 1 - cos as
// |x_i/|x_i| - x_{i-1}/|x_{i-1}||^2 / 2.
//
// Every mbarrier wait is bounded (kWaitLimitNs); on expiry the kernel sets
// ART_STATUS_TIMEOUT, the producer waits for its own copies in flight, and
// the CTA returns.
#pragma once

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

template <bool kBF16, int D, int G>
struct Cfg {
    using E = Elem<kBF16>;
    static constexpr int GQ = G;                 // query heads per KV head
    static constexpr int ELT = E::kBytes;
    static constexpr int DD = D;
    static constexpr int ROWB = D * ELT;         // bytes of one K or V row
    static constexpr int CB = ROWB / 8 <= 32 ? 8 : 16;  // bytes of a row one lane reads
    static constexpr int EPC = CB / ELT;         // elements per chunk
    static constexpr int E2 = EPC / 2;           // packed pairs per chunk
    static constexpr int LPR = ROWB / CB;        // lanes covering one row
    static constexpr int RPW = 32 / LPR;         // rows per warp instruction
    static constexpr int RW = kBK / kNWC;        // rows per consumer warp per block
    static constexpr int NI = RW / RPW;          // warp instructions per block
    static constexpr int NV = NI * G;            // partial scores per lane
    static constexpr int NVP = pow2ceil(imax(NV, LPR));
    static constexpr int QB = (int)align_up((size_t)G * D * ELT, 16);
    static constexpr int KVB = kBK * ROWB;       // bytes of K (or V) of one block
    static constexpr int SLOT = 2 * KVB + QB;
    static constexpr int SPL = (G * kMaxProbe + 31) / 32;  // probe slots per stat lane
    static constexpr int PART_F = 2 * kNWC * RPW * G * kMaxProbe;
    static constexpr bool LAG = G <= 4;          // decision one block behind (register budget)
    static_assert(LPR >= 8 && LPR <= 32 && EPC >= 2 && EPC <= 8, "row must be 128..512 bytes");
    static_assert(RW % RPW == 0 && NI >= 1, "rows per warp");
    static_assert(32 % RW == 0, "softmax lane groups");
    static_assert(G >= 1 && G <= 8, "group size");
};

struct SlotMeta {
    int item, pos, n, c, nvalid, kind, b, g, has0, pad0, pad1, pad2;
};

struct Ctrl {
    int dec[2];
    int stop_item;
    int abort;
    SlotMeta info[2];  // item and position of each published partial
};

struct Layout {
    size_t meta, bars, part, plb, pmb, wmax, scr, eacc, sh, ptab, ctrl, total;
};

template <class C>
__host__ __device__ inline Layout make_layout(int stages) {
    constexpr int G = C::GQ;
    Layout L;
    size_t o = (size_t)stages * C::SLOT;
    L.meta = o;
    o += (size_t)stages * sizeof(SlotMeta);
    o = align_up(o, 16);
    L.bars = o;
    o += (size_t)(2 * stages + 5) * sizeof(uint64_t);
    o = align_up(o, 16);
    L.part = o;  // [2][NWC][RPW][G][kMaxProbe] probe partials
    o += (size_t)C::PART_F * sizeof(float);
    L.plb = o;  // [2][NWC][G] per-warp block sums
    o += (size_t)2 * kNWC * G * sizeof(float);
    L.pmb = o;  // [2][G] block maxima
    o += (size_t)2 * G * sizeof(float);
    L.wmax = o;  // [NWC][G] per-warp maxima of the block being processed
    o += (size_t)kNWC * G * sizeof(float);
    L.scr = o;  // [NWC][G][RW] scores, then weights
    o += (size_t)kNWC * G * C::RW * sizeof(float);
    o = align_up(o, 16);
    L.eacc = o;  // per consumer warp: [G][D] output sums, then [G] weight sums
    o += (size_t)kNWC * (G * C::DD + G) * sizeof(float);
    o = align_up(o, 16);
    L.sh = o;  // [3][G] statistics warp scratch
    o += (size_t)3 * G * sizeof(float);
    o = align_up(o, 16);
    L.ptab = o;
    o += (size_t)2 * C::LPR * sizeof(int);
    o = align_up(o, 16);
    L.ctrl = o;
    o += sizeof(Ctrl);
    L.total = align_up(o, 128);
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
// Returns false when the CTA is aborting or the wait exceeded kWaitLimitNs.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, Ctrl* ctrl, WsHeader* hdr) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        int stop = ld_volatile_shared(&ctrl->abort);
        if (!stop && (threadIdx.x & 31) == 0 && global_ns() - t0 > kWaitLimitNs) {
            st_volatile_shared(&ctrl->abort, 1);
            atomicOr(&hdr->status, ART_STATUS_TIMEOUT);
            stop = 1;
        }
        if (__any_sync(0xffffffffu, stop)) return false;
    }
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <class C, bool kART>
__device__ void producer_warp(const Params& p, unsigned char* ring, SlotMeta* meta, uint64_t* full,
                              uint64_t* empty, Ctrl* ctrl) {
    constexpr int G = C::GQ;
    const int lane = threadIdx.x & 31;
    int slot = 0;
    uint32_t round = 0;
    bool have_slot = false;
    unsigned long long issued = 0;
    bool ok = true;

    auto acquire = [&]() -> bool {
        if (have_slot) return true;
        if (!wait_bounded(&empty[slot], (round & 1u) ^ 1u, ctrl, p.hdr)) return false;
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
    auto emit = [&](int kind, int item, int b, int g) -> bool {
        if (!acquire()) return false;
        if (lane == 0) {
            SlotMeta& mt = meta[slot];
            mt.item = item; mt.pos = 0; mt.n = 0; mt.c = 0; mt.nvalid = 0; mt.kind = kind;
            mt.b = b; mt.g = g; mt.has0 = 0;
            mbar_arrive(&full[slot]);
        }
        __syncwarp();
        advance();
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
                const int cj = __shfl_sync(0xffffffffu, c, j);
                const int nvj = __shfl_sync(0xffffffffu, nvalid, j);
                const int npj = __shfl_sync(0xffffffffu, npv, j);
                const int badj = __shfl_sync(0xffffffffu, bad, j);
                const int r0j = __shfl_sync(0xffffffffu, r0, j);
                int pgj[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) pgj[k] = __shfl_sync(0xffffffffu, pg[k], j);
                if (badj) {
                    if (lane == 0) atomicOr(&p.hdr->status, ART_STATUS_BAD_PAGE);
                    if (!(ok = emit(kSlotFail, item, b, g))) break;
                    item_done = true;
                    break;
                }
                const int posj = base + j;
                const bool with_q = (posj == 0);
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
                        const char* src = static_cast<const char*>(p.q) + ((size_t)b * p.Hq + (size_t)g * G) * C::ROWB;
                        bulk_g2s(dst + 2 * C::KVB, src, (uint32_t)(G * C::ROWB), &full[slot]);
                    }
                }
                __syncwarp();
                advance();
            }
            if (!ok) break;
        }
        if (!ok) break;
    }

    if (!ok) {
        // aborting: wait (bounded) for this CTA's own copies still in flight
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
// statistics warp (ART only)
// ---------------------------------------------------------------------------
template <class C>
__device__ void stat_warp(const Params& p, const float* part, const float* plb, const float* pmb, float* sh,
                          uint64_t* part_full, uint64_t* dec_bar, Ctrl* ctrl) {
    constexpr int G = C::GQ;
    constexpr int SPL = C::SPL;
    constexpr int RPW = C::RPW;
    const int lane = threadIdx.x & 31;
    const int m = p.m;
    const int GM = G * m;
    // the probe slot of each (lane, j): head and column rank
    int hs[SPL], ss[SPL];
#pragma unroll
    for (int j = 0; j < SPL; ++j) {
        const int k = lane + 32 * j;
        hs[j] = k < GM ? k / m : -1;
        ss[j] = k < GM ? k - (k / m) * m : 0;
    }
    float Mh = -INFINITY, Lh = 0.f;  // running max / sum of head `lane` (lanes < G)
    float X[SPL], dl[SPL];
    float nprev = 0.f;
    int counter = 0, seen0 = 0;
    int stopped_item = -1;
    auto reset = [&]() {
        Mh = -INFINITY;
        Lh = 0.f;
#pragma unroll
        for (int j = 0; j < SPL; ++j) X[j] = 0.f;
        nprev = 0.f;
        counter = 0;
        seen0 = 0;
    };
    reset();
    for (int v = 0;; ++v) {
        const int vb = v & 1;
        if (!wait_bounded(&part_full[vb], (uint32_t)(v >> 1) & 1u, ctrl, p.hdr)) return;
        const SlotMeta info = ctrl->info[vb];
        if (info.kind == kSlotEnd) return;
        int dec = kStop;
        if (info.kind != kSlotBlock) {
            if (lane == 0) p.blocks_used[info.item] = info.kind == kSlotFail ? -1 : 0;
            reset();
        } else if (info.item == stopped_item) {
            dec = kDiscard;  // computed ahead of the decision that stopped its item
        } else {
            if (info.pos == 0) reset();
            // per head: block sum over the warps, new running max and sum
            if (lane < G) {
                const float mb = pmb[vb * G + lane];
                float lb = 0.f;
#pragma unroll
                for (int w = 0; w < kNWC; ++w) lb += plb[(vb * kNWC + w) * G + lane];
                const float Mn = fmaxf(Mh, mb);
                const float a = exp2f(Mh - Mn);
                const float bw = exp2f(mb - Mn);
                const float Ln = a * Lh + bw * lb;
                sh[lane] = bw;
                sh[G + lane] = lb;
                sh[2 * G + lane] = Ln;
                Mh = Mn;
                Lh = Ln;
            }
            __syncwarp();
            const float* pp = part + (size_t)vb * kNWC * RPW * G * kMaxProbe;
            float sx2 = 0.f, sdd = 0.f;
#pragma unroll
            for (int j = 0; j < SPL; ++j) {
                dl[j] = 0.f;
                const int h = hs[j];
                if (h >= 0) {
                    float pb = 0.f;
#pragma unroll
                    for (int w = 0; w < kNWC * RPW; ++w) pb += pp[(w * G + h) * kMaxProbe + ss[j]];
                    const float d = sh[h] * (pb - sh[G + h] * X[j]) / sh[2 * G + h];
                    dl[j] = d;
                    const float x = X[j] + d;
                    sx2 += x * x;
                    sdd += d * (2.f * X[j] + d);
                }
            }
            sx2 = warp_sum(sx2);
            sdd = warp_sum(sdd);
            const float ni = sqrtf(sx2);
            const float dn = sdd / (ni + nprev);
            bool stable = false;
            if (info.pos >= 1) {
                float su2 = 0.f;
                const float cx = dn / (ni * nprev);
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    if (hs[j] >= 0) {
                        const float u = dl[j] / ni - X[j] * cx;
                        su2 += u * u;
                    }
                }
                su2 = warp_sum(su2);
                const float dmag = fabsf(dn) / nprev;
                const float ddir = 0.5f * su2;
                stable = nprev > 0.f && ni > 0.f && isfinite(nprev) && isfinite(ni) && isfinite(dmag) &&
                         isfinite(ddir) && dmag < p.eps_mag && ddir < p.eps_dir;
            }
            counter = stable ? counter + 1 : 0;
            if (info.c == 0) seen0 = 1;
            const bool stop = ((counter >= p.patience) && (seen0 || !info.has0)) || (info.pos == info.n - 1);
#pragma unroll
            for (int j = 0; j < SPL; ++j) X[j] += dl[j];
            nprev = ni;
            dec = stop ? kStop : kContinue;
            if (stop) {
                stopped_item = info.item;
                if (lane == 0) {
                    p.blocks_used[info.item] = info.pos + 1;
                    st_volatile_shared(&ctrl->stop_item, info.item);
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            ctrl->dec[vb] = dec;
            mbar_arrive(&dec_bar[vb]);
        }
        __syncwarp();
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
    int stopped_item = -1;

    auto cbar_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(cbar);
        const bool r = wait_bounded(cbar, cbph, ctrl, p.hdr);
        cbph ^= 1u;
        return r;
    };
    auto release = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
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
        if (lane == 0) mbar_arrive(&part_full[vb]);
        return v++;
    };
    auto wait_dec = [&](int rec) -> int {
        if (!wait_bounded(&dec_bar[rec & 1], (uint32_t)(rec >> 1) & 1u, ctrl, p.hdr)) return -1;
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
        float* mine = eacc + (size_t)w * (G * D + G);  // this warp's [G][D] sums, then [G] weights
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
                num += eacc[(size_t)ww * (G * D + G) + idx];
                den += eacc[(size_t)ww * (G * D + G) + G * D + h];
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
        if (!wait_bounded(&full[slot], round & 1u, ctrl, p.hdr)) return;
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
            if (h < G && rl == 0) wmax[w * G + h] = mx;
        }
        named_bar_sync(1, kNWC * 32);
#pragma unroll
        for (int k = 0; k < (G * kNWC + 31) / 32; ++k) {
            const int idx = k * 32 + lane;
            const int h = idx / kNWC, ww = idx % kNWC;
            float mx = h < G ? wmax[ww * G + h] : -INFINITY;
#pragma unroll
            for (int o = kNWC / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
                if (hh / (32 / kNWC) == k) mbN[hh] = __shfl_sync(0xffffffffu, mx, (hh % (32 / kNWC)) * kNWC);
        }
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
            float* pp = part + (((size_t)vb * kNWC + w) * RPW + half) * G * kMaxProbe;
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                if ((my_mask >> e) & 1u) {
                    const int s = my_base + __popc(my_mask & ((1u << e) - 1u));
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float lo, hi;
                        up2(tN[h][e >> 1], lo, hi);
                        pp[h * kMaxProbe + s] = (e & 1) ? hi : lo;
                    }
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h) plb[(vb * kNWC + w) * G + h] = lbN[h];
            }
            if (w == 0 && lane == 0) {
#pragma unroll
                for (int h = 0; h < G; ++h) pmb[vb * G + h] = mbN[h];
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
// the kernel
// ---------------------------------------------------------------------------
template <bool kBF16, int D, int G, bool kART>
__global__ void __launch_bounds__(kThreads, 1) art_decode_kernel(const Params p) {
    using C = Cfg<kBF16, D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    const Layout L = make_layout<C>(p.stages);
    unsigned char* ring = smem;
    SlotMeta* meta = reinterpret_cast<SlotMeta*>(smem + L.meta);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + p.stages;
    uint64_t* part_full = empty + p.stages;
    uint64_t* dec_bar = part_full + 2;
    uint64_t* cbar = dec_bar + 2;
    int* pmask = reinterpret_cast<int*>(smem + L.ptab);
    int* pbase = pmask + C::LPR;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + L.ctrl);

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kNWC);
        }
        mbar_init(&part_full[0], kNWC);
        mbar_init(&part_full[1], kNWC);
        mbar_init(&dec_bar[0], 1);
        mbar_init(&dec_bar[1], 1);
        mbar_init(cbar, kNWC);
        ctrl->stop_item = -1;
        ctrl->abort = 0;
        ctrl->dec[0] = ctrl->dec[1] = 0;
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
    __syncthreads();

    const int warp = tid >> 5;
    if (warp == kProducerWarp) {
        producer_warp<C, kART>(p, ring, meta, full, empty, ctrl);
    } else if (warp == kStatWarp) {
        if (kART)
            stat_warp<C>(p, reinterpret_cast<const float*>(smem + L.part), reinterpret_cast<const float*>(smem + L.plb),
                         reinterpret_cast<const float*>(smem + L.pmb), reinterpret_cast<float*>(smem + L.sh),
                         part_full, dec_bar, ctrl);
    } else {
        consumer_warps<C, kART>(p, ring, meta, full, empty, part_full, dec_bar, cbar, L, smem, pmask, pbase, ctrl);
    }
}

// Largest ring depth (2..8 slots) that fits one CTA per SM.
template <class C>
inline int pick_stages(int smem_per_block) {
    for (int s = 8; s >= 2; --s)
        if ((int)make_layout<C>(s).total <= smem_per_block) return s;
    return 0;
}

template <bool kBF16, int D, int G, bool kART>
cudaError_t launch_main(Params p, cudaStream_t stream, int force_stages, LaunchInfo* li) {
    using C = Cfg<kBF16, D, G>;
    auto kern = art_decode_kernel<kBF16, D, G, kART>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 0, smem_blk = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    const int stages = force_stages >= 2 && force_stages <= 8 ? force_stages : pick_stages<C>(smem_blk);
    if (stages == 0) return cudaErrorInvalidConfiguration;
    const size_t smem = make_layout<C>(stages).total;
    if ((int)smem > smem_blk) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    int occ = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem)) != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    p.stages = stages;
    int grid = sms * occ;
    if (grid > p.num_items) grid = p.num_items;
    if (li) { li->grid = grid; li->stages = stages; li->smem = smem; li->ctas_per_sm = occ; }
    kern<<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace art

#define ART_INSTANTIATE(BF, D, G)                                                                           \
    template cudaError_t art::launch_main<BF, D, G, true>(art::Params, cudaStream_t, int, art::LaunchInfo*); \
    template cudaError_t art::launch_main<BF, D, G, false>(art::Params, cudaStream_t, int, art::LaunchInfo*);
