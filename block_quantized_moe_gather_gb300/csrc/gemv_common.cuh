// Device helpers shared by the GEMV kernels (gemv.cu, gemv_stream.cu):
// bulk copies and bounded mbarrier waits, cluster/DSMEM access, the
// mma.sync m16n8k16 fragment MMA and the bit-field to fp16 conversions.
#pragma once

#include "moe_internal.cuh"

namespace bq {
namespace gemv {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(100000u) : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for phase `parity` of an mbarrier: false after the limit
// (BQ_DEV_WAIT_TIMEOUT recorded).
// Between tests the warp sleeps, 32 ns doubling up to 512 ns, so that warps
// waiting for their first slab leave the issue slots to warps with data.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    unsigned ns = 32;
    while (!mbar_try(bar, parity)) {
        __nanosleep(ns);
        ns = ns < 512 ? 2 * ns : ns;
        if (global_ns() - t0 > kWaitLimitNs) {
            bq::set_device_error(status, BQ_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 bytes at shared address `addr` of CTA `rank` of this cluster.
__device__ __forceinline__ float4 ld_dsmem(uint32_t addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Exact small integers from bit fields: a field at bit J of each 16-bit lane
// ORed into the mantissa of 2^(10-J) has weight 1; subtracting 2^(10-J)
// leaves its value.
template <int J>
__device__ __forceinline__ __half2 field_h2(uint32_t w, uint32_t mask) {
    constexpr uint32_t e = (uint32_t)(25 - J) << 10;   // biased exponent of 2^(10-J)
    return __hsub2(bq::u32_as_h2((w & (mask << J)) | e | (e << 16)), bq::u32_as_h2(e | (e << 16)));
}

// ---- Q2_K code pairs as fp16 subnormals.  Sub-block word layout: value 2p
// in bits 2p..2p+1 of the low 16-bit lane, value 2p+1 in the same bits of the
// high lane (p = 0..7); pairs 5-7 are taken from the word shifted right by
// 10.  Pair p sits at bit J(p) of its lane, where ANDing it out leaves the
// fp16 bit pattern of q * 2^(J - 24) (exponent field 0).
__host__ __device__ constexpr int q2_j(int p) { return p < 5 ? 2 * p : 2 * (p - 5); }

template <int P>
__device__ __forceinline__ uint32_t q2_sub(uint32_t w, uint32_t wh) {
    return (P < 5 ? w : wh) & (0x00030003u << q2_j(P));
}

// The activation factor 2^-J of element e (0..3) of MMA step s: elements 0-1
// meet pair 2(s % 4), elements 2-3 pair 2(s % 4) + 1 of the step's sub-block.
__host__ __device__ constexpr int q2_step_j(int s, int e) { return q2_j(2 * (s & 3) + (e >> 1)); }

}  // namespace gemv
}  // namespace bq
