// Device-side building blocks for the sm_103a MXFP4 weight-streaming kernels:
// mbarriers with bounded waits, TMA (bulk and tiled-tensor) copies, the
// legacy warp MMA, and the E2M1 -> f16 unpack.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mxfp4 {

// Every spin-wait gives up after this many nanoseconds of %globaltimer. A
// test-only build shortens it (see MXFP4_TEST_WITHHOLD_STAGE).
#ifndef MXFP4_WAIT_LIMIT_NS
#define MXFP4_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t kWaitLimitNs = MXFP4_WAIT_LIMIT_NS;

// Test-only builds (compiled with MXFP4_TEST_WITHHOLD_STAGE, never the
// product library): the producer of CTA 0 withholds its first weight stage
// (no copy, no arrive), so the consumers' bounded wait on it runs out. This
// exercises the timeout path - status word, wind-down, a usable context -
// without any fault.
__device__ __forceinline__ bool withhold_stage(uint32_t index) {
#ifdef MXFP4_TEST_WITHHOLD_STAGE
    return blockIdx.x == 0 && index == 0;
#else
    (void)index;
    return false;
#endif
}

// Bits of the per-device status word.
constexpr unsigned kStatusTimeout = 1u;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Ends an mbarrier's life so its memory may be used for anything else
// (including a new mbarrier).
__device__ __forceinline__ void mbar_inval(uint32_t bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// One potentially blocking test of the phase (the hardware's own time
// limit applies; a suspend-time hint measured no better).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking tests of two, three or four mbarrier phases in one go: the
// tests are independent, so they cost one shared-memory round trip, not one
// each (each is about 90 ns on GB300 with the copy engine and tensor cores
// busy). True if every phase has completed.
__device__ __forceinline__ bool mbar_test2(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q1, q2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%1], %2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%3], %4;\n\t"
        "and.pred q1, q1, q2;\n\tselp.u32 %0, 1, 0, q1;\n\t}"
        : "=r"(ok)
        : "r"(b1), "r"(p1), "r"(b2), "r"(p2)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test3(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2, uint32_t b3,
                                           uint32_t p3) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q1, q2, q3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%1], %2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%3], %4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q3, [%5], %6;\n\t"
        "and.pred q1, q1, q2;\n\tand.pred q1, q1, q3;\n\tselp.u32 %0, 1, 0, q1;\n\t}"
        : "=r"(ok)
        : "r"(b1), "r"(p1), "r"(b2), "r"(p2), "r"(b3), "r"(p3)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test4(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2, uint32_t b3,
                                           uint32_t p3, uint32_t b4, uint32_t p4) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q1, q2, q3, q4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q1, [%1], %2;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q2, [%3], %4;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q3, [%5], %6;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 q4, [%7], %8;\n\t"
        "and.pred q1, q1, q2;\n\tand.pred q3, q3, q4;\n\tand.pred q1, q1, q3;\n\tselp.u32 %0, 1, 0, q1;\n\t}"
        : "=r"(ok)
        : "r"(b1), "r"(p1), "r"(b2), "r"(p2), "r"(b3), "r"(p3), "r"(b4), "r"(p4)
        : "memory");
    return ok != 0;
}

// Where a bounded wait reports: the per-device status word, and a per-CTA
// abort flag in shared memory. Once one wait of a CTA has given up, every
// later wait of that CTA fails at once, so the CTA winds down in one limit
// rather than one limit per remaining wait.
struct WaitCtx {
    unsigned* status;
    volatile int* abort;
};

__device__ __forceinline__ void record_timeout(const WaitCtx& w) {
    *w.abort = 1;
    atomicOr(w.status, kStatusTimeout);
}

// Waits until the phase with the given parity has completed. Returns false
// if the CTA has aborted or the wait takes longer than the limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (*w.abort) return false;
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_timeout(w);
            return false;
        }
    }
}

// Adds v to a device word with release semantics at GPU scope: the calling
// thread's earlier writes are visible to whoever observes the new value.
__device__ __forceinline__ void atom_add_release_gpu(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until the device word at p is at least want (counted by other CTAs
// of the grid, which must all be resident). Same limits as mbar_wait. No
// sleep between reads: each acquire load is already an L2 round trip, and
// a sleep measured as 1-2 us of lag between the last count and the waiters.
__device__ __forceinline__ bool wait_global_at_least(const unsigned* p, unsigned want, const WaitCtx& w) {
    if (ld_acquire_gpu(p) >= want) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (*w.abort) return false;
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ld_acquire_gpu(p) >= want) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_timeout(w);
            return false;
        }
    }
}

// Waits until the shared word at addr holds want (written by another warp of
// the CTA). Same limits as mbar_wait.
__device__ __forceinline__ uint32_t lds_u32_volatile(uint32_t a) {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ void sts_u32_volatile(uint32_t a, uint32_t v) {
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ bool wait_shared_value(uint32_t addr, uint32_t want, const WaitCtx& w) {
    if (lds_u32_volatile(addr) == want) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (*w.abort) return false;
#pragma unroll 1
        for (int i = 0; i < 32; ++i) {
            __nanosleep(32);
            if (lds_u32_volatile(addr) == want) return true;
        }
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_timeout(w);
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t atom_add_shared(uint32_t a, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
    return old;
}

// ------------------------------------------- programmatic dependent launch
// Lets the next kernel of the stream be scheduled before this one ends (its
// CTAs become resident as SMs free up).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the previous kernel of the stream has completed and its
// writes are visible (a no-op when this kernel was not launched early).
__device__ __forceinline__ void pdl_wait_previous() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Atomic add on a shared word of any CTA of the cluster (relaxed); returns
// the old value.
__device__ __forceinline__ uint32_t atom_add_cluster(uint32_t cluster_addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(cluster_addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Makes this thread's earlier writes (and those ordered before them, e.g.
// by a warp barrier) visible cluster-wide before its later writes.
__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

// Whole-cluster barrier (every thread of every CTA).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2D tiled tensor load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 3D tiled tensor load (coordinates innermost first), completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// 5D tiled tensor load (coordinates innermost first), completing on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            int32_t c3, int32_t c4, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "l"(policy)
        : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// The same bulk copy with the default L2 policy (for data that many CTAs
// read, such as activations).
__device__ __forceinline__ void bulk_load_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory
// before its later bulk (async-proxy) copies into it.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------- shared-memory loads
// Explicit ld.shared on 32-bit shared addresses (a generic pointer into
// shared memory would go through the slower generic path). Volatile so they
// stay ordered after the mbarrier waits that publish the data.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ uint64_t lds64_pair(uint32_t a) {
    uint64_t v;
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ void lds128_pairs(uint32_t a, uint64_t& lo, uint64_t& hi) {
    asm volatile("ld.shared.v2.b64 {%0,%1}, [%2];" : "=l"(lo), "=l"(hi) : "r"(a));
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// ------------------------------------------------------- warp-level math
// Four 8x8 b16 matrices from shared memory (lane l supplies the row address
// of matrix l/8, row l%8); lane l receives 4 bytes of row l/4 of each.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// The two chained m16n8k16 products of one 32-block: A holds the 16 rows'
// f16 weights (k permuted consistently with B), B the 8 columns' f16
// activations, no accumulator input. The result comes back as the pairs
// {d0, d1} (row g, columns 2t and 2t+1) and {d2, d3} (row g+8), each in
// one 64-bit register pair for the packed f32x2 arithmetic below.
__device__ __forceinline__ void mma_f16_k32(uint64_t& d01, uint64_t& d23, const uint32_t (&ga)[4],
                                            const uint32_t (&gb)[4], const uint4& x) {
    asm("{\n\t.reg .f32 t0, t1, t2, t3;\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {t0,t1,t2,t3}, {%2,%3,%4,%5}, {%10,%11}, "
        "{0f00000000,0f00000000,0f00000000,0f00000000};\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {t0,t1,t2,t3}, {%6,%7,%8,%9}, {%12,%13}, "
        "{t0,t1,t2,t3};\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t}"
        : "=l"(d01), "=l"(d23)
        : "r"(ga[0]), "r"(gb[0]), "r"(ga[1]), "r"(gb[1]), "r"(ga[2]), "r"(gb[2]), "r"(ga[3]), "r"(gb[3]),
          "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
}

// ------------------------------------------------------ packed f32 pairs
// Blackwell issues two f32 multiplies or FMAs per instruction on a register
// pair; a pair travels as one 64-bit value (low half = first element).
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f32x2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Two E8M0 scale bytes (bits 0-7 and 8-15 of v) -> bf16x2 {2^(s0-127),
// 2^(s1-127)}: bf16 holds every such power of two exactly (s = 0 is the
// subnormal 2^-127).
__device__ __forceinline__ uint32_t e8m0x2_to_bf16x2(uint32_t v) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.bf16x2.ue8m0x2 %0, lo;\n\t}"
        : "=r"(r)
        : "r"(v));
    return r;
}

// Four bytes of packed E2M1 pairs -> four f16x2 words (byte i -> out[i]);
// the low nibble of each byte becomes the low half of its word.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t v, uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                                uint32_t& o3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
        : "r"(v));
}

// 2^e as float32 for e in [-149, 127], exact.
__device__ __forceinline__ float exp2_int(int e) {
    return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(1 << (e + 149));
}

}  // namespace mxfp4
