// art_common.cuh -- shared definitions of the ART decode-attention kernels:
// launch parameters, workspace layout, and thin wrappers around the sm_100+
// PTX used for the shared-memory ring (mbarrier, cp.async.bulk).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "art.h"

namespace art {

constexpr int kBK = 64;          // tokens per ART block (the unit of the stability test)
constexpr int kMaxProbe = 32;    // probe entries per query head
// CTA layout: consumer warps 0..NWC-1, then the producer warp, then the statistics warp.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded waits give up after 1 s

// Item flags written by the plan kernel.
constexpr int kItemHas0 = 1;     // logical block 0 is in the visit list
constexpr int kItemBad = 2;      // the item's device data failed a check

// Slot kinds written by the producer into the ring metadata.
// kSlotPad: an entry without data that gives the second consumer group its
// share of a one-block item.
enum SlotKind : int { kSlotBlock = 0, kSlotEmpty = 1, kSlotFail = 2, kSlotEnd = 3, kSlotPad = 4 };

struct WsHeader {
    unsigned int claim;      // next position of `order` to hand out
    unsigned int plan_done;  // plan CTAs that have finished
    int status;              // ART_STATUS_* bits
    int check_code;          // first failed internal check (0 = none)
    int check_info[4];       // its details
    unsigned int uclaim;     // unit path: next unit to hand out
    int n_regular;           // unit path: units of the visit lists (the fix units follow)
    int n_units;             // unit path: all units
    int ck;                  // unit path: ART blocks per unit, chosen by the plan kernel
    int pad[4];
};

// Host: keeps the text of a failed CUDA call for art_last_cuda_error and returns ART_ERR_LAUNCH.
int cuda_fail(cudaError_t e);

// Records the first failed internal consistency check (ART_STATUS_INTERNAL).
__device__ __forceinline__ void record_check(WsHeader* hdr, int code, int a, int b, int c) {
    if (atomicCAS(&hdr->check_code, 0, code) == 0) {
        hdr->check_info[0] = a;
        hdr->check_info[1] = b;
        hdr->check_info[2] = c;
        hdr->check_info[3] = (int)blockIdx.x;
    }
    atomicOr(&hdr->status, ART_STATUS_INTERNAL);
}
static_assert(sizeof(WsHeader) == 64, "workspace header is 64 bytes");

struct ItemInfo {
    int n;      // listed blocks
    int flags;  // kItemHas0 | kItemBad
};

struct Params {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* visit;  // may be null (natural order)
    const int32_t* probe;  // may be null for the dense twin
    void* out;
    int32_t* blocks_used;  // may be null for the dense twin
    WsHeader* hdr;
    const int32_t* order;
    const ItemInfo* info;
    int B, Hq, Hkv, Ps, max_pages, max_visit, m, num_pages, num_items, stages;
    int tma3d;  // tensor-core path: one 3-D copy per page (else one 2-D copy per 128-byte column half)
    float eps_mag, eps_dir;
    int patience;
    int ph;  // query heads 0 .. ph-1 of a group form the probe
    // Bounded waits give up after wait_ns (kWaitLimitNs unless the test hook below is
    // set); a warp's final drain of its own copies always allows kWaitLimitNs.
    unsigned long long wait_ns;
    // Test hook of the failure path: the consumer warps first wait on a barrier that
    // nothing completes, so every warp of the CTA gives up at one of its bounded waits
    // (none reaches a named barrier) and the call ends with ART_STATUS_TIMEOUT.
    int stall;
};

// Launch geometry chosen for one call.
struct LaunchInfo {
    int grid;
    int stages;
    size_t smem;
    int ctas_per_sm;
};

// Workspace: header, then ItemInfo[num_items], then the claim order int32[num_items].
inline size_t workspace_bytes_for(int num_items) {
    return sizeof(WsHeader) + (size_t)num_items * (sizeof(int32_t) + sizeof(ItemInfo));
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// one arrive from the lanes where `pred` holds (typically one lane), without a branch
__device__ __forceinline__ void mbar_arrive_if(bool pred, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %0, 0;\n\t"
        "@q mbarrier.arrive.shared::cta.b64 _, [%1];\n\t}" ::"r"((int)pred),
        "r"(smem_addr(bar))
        : "memory");
}

// Predicated shared-memory stores: lanes store or not without a divergent branch.
__device__ __forceinline__ void st_shared_if(bool pred, int* p, int v) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %0, 0;\n\t"
        "@q st.shared.b32 [%1], %2;\n\t}" ::"r"((int)pred),
        "r"(smem_addr(p)), "r"(v)
        : "memory");
}
__device__ __forceinline__ void st_shared_if(bool pred, float* p, float v) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %0, 0;\n\t"
        "@q st.shared.f32 [%1], %2;\n\t}" ::"r"((int)pred),
        "r"(smem_addr(p)), "f"(v)
        : "memory");
}
__device__ __forceinline__ void st_shared_if(bool pred, uint32_t addr, float x, float y) {  // addr 8-byte aligned
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %0, 0;\n\t"
        "@q st.shared.v2.f32 [%1], {%2, %3};\n\t}" ::"r"((int)pred),
        "r"(addr), "f"(x), "f"(y)
        : "memory");
}
__device__ __forceinline__ void st_shared_if(bool pred, uint32_t addr, float x) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %0, 0;\n\t"
        "@q st.shared.f32 [%1], %2;\n\t}" ::"r"((int)pred),
        "r"(addr), "f"(x)
        : "memory");
}
__device__ __forceinline__ void st_shared_if(bool pred, float* p, float x, float y) {  // p 8-byte aligned
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %0, 0;\n\t"
        "@q st.shared.v2.f32 [%1], {%2, %3};\n\t}" ::"r"((int)pred),
        "r"(smem_addr(p)), "f"(x), "f"(y)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Non-blocking test of a phase (no suspension).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` waiting for the
// phase (it resumes as soon as the phase completes) instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bulk copy global -> this CTA's shared memory, completing on `bar` (tx bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Named barrier among a set of consumer warps (ids 1..15; 0 is __syncthreads).
// bar.sync is a warp-aligned instruction: the warp is reconverged first.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic; each half is an IEEE fp32 op).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void up2(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Tiled tensor copy (2-D tensor map, box written with the map's swizzle) global -> shared,
// completing on `bar`. x: element offset of the innermost dimension (16-byte aligned), y: row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// two bf16 products, round to nearest
__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ldmatrix / movmatrix / mma.sync (bf16 in, fp32 accumulate) fragments.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
// d[0..3] += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// two fp32 -> bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf16_lo_f(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ int ld_volatile_shared(const int* p) { return *(const volatile int*)p; }
__device__ __forceinline__ void st_volatile_shared(int* p, int v) { *(volatile int*)p = v; }

// ---------------------------------------------------------------------------
// element handling. A lane reads CB bytes (one "chunk") of a K/V/q row and
// turns them into packed fp32 pairs (elements 2i, 2i+1 of the chunk).
// ---------------------------------------------------------------------------
template <bool kBF16>
struct Elem;

template <>
struct Elem<true> {
    static constexpr int kBytes = 2;
    template <int CB>
    __device__ __forceinline__ static void load_pairs(const unsigned char* src, uint64_t* f2) {
        if constexpr (CB == 8) {
            const uint2 u = *reinterpret_cast<const uint2*>(src);
            f2[0] = pk2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
            f2[1] = pk2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
        } else {
            const uint4 u = *reinterpret_cast<const uint4*>(src);
            f2[0] = pk2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
            f2[1] = pk2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
            f2[2] = pk2(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u));
            f2[3] = pk2(__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
        }
    }
    // round to nearest even
    __device__ __forceinline__ static void store(void* base, size_t idx, float x) {
        uint32_t u = __float_as_uint(x);
        uint32_t r = (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
        if ((u & 0x7fffffffu) > 0x7f800000u) r = 0x7fc0u;  // NaN stays NaN
        static_cast<uint16_t*>(base)[idx] = static_cast<uint16_t>(r);
    }
};

template <>
struct Elem<false> {
    static constexpr int kBytes = 4;
    template <int CB>
    __device__ __forceinline__ static void load_pairs(const unsigned char* src, uint64_t* f2) {
        if constexpr (CB == 8) {
            const uint2 u = *reinterpret_cast<const uint2*>(src);
            f2[0] = pk2(__uint_as_float(u.x), __uint_as_float(u.y));
        } else {
            const uint4 u = *reinterpret_cast<const uint4*>(src);
            f2[0] = pk2(__uint_as_float(u.x), __uint_as_float(u.y));
            f2[1] = pk2(__uint_as_float(u.z), __uint_as_float(u.w));
        }
    }
    __device__ __forceinline__ static void store(void* base, size_t idx, float x) {
        static_cast<float*>(base)[idx] = x;
    }
};

}  // namespace art
