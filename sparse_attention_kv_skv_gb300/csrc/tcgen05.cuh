// Blackwell (sm_100 family) tensor-core primitives used by the attention
// consumer: shared-memory matrix descriptors, the tcgen05 MMA (bf16 x bf16 ->
// fp32, accumulator in tensor memory), tensor-memory allocation and loads /
// stores, bounded mbarrier waits, plus the TMA row gather and cluster (CTA
// pair) operations the attention pipeline uses.  Written from the PTX
// ISA's description of these instructions; no vendor library code.
#pragma once

#include <cstdint>

namespace skv {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Canonical K-major operand layout without swizzle, for a tile of R rows
// (M or N) by Kd bf16 elements: 8 x 16-byte "core matrices" (8 rows of 8
// elements), consecutive along K at LBO = 128 bytes, 8-row groups at
// SBO = Kd / 8 * 128 bytes.  Byte offset of the 16-byte chunk c (elements
// 8c..8c+7) of row r:
__host__ __device__ constexpr uint32_t kmajor_chunk_offset(uint32_t r, uint32_t c, uint32_t Kd)
{
    return (r >> 3) * (Kd / 8 * 128u) + c * 128u + (r & 7u) * 16u;
}
__host__ __device__ constexpr uint32_t kmajor_elem_offset(uint32_t r, uint32_t k, uint32_t Kd)
{
    return kmajor_chunk_offset(r, k >> 3, Kd) + (k & 7u) * 2u;
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// (K-direction) and stride (8-row-group) byte offsets, descriptor version 1,
// no swizzle.  The MMA's k-th step of 16 elements starts 256 bytes further.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr, uint32_t Kd)
{
    const uint32_t lbo = 128u, sbo = Kd / 8 * 128u;
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// The same canonical layout seen as an MN-major operand: a buffer of Kr
// rows of Nd contiguous elements (row = one k, elements along M/N), stored as
// core matrices of 8 k-rows x 16 bytes (8 elements along M/N), consecutive
// along M/N at 128 bytes, 8-row k groups at `kgroup` bytes.  For an MN-major
// operand the descriptor's stride offset (SBO) is the M/N-direction core
// matrix stride and its leading offset (LBO) the K-direction group stride --
// the reverse of the K-major case.  A K-major tile of (keys x dims) is
// exactly such a buffer for a product whose M/N runs over dims and whose K
// runs over keys (kgroup = its 8-row-group stride).  The MMA's k-th step of
// 16 rows starts 2 * kgroup bytes further.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t saddr, uint32_t kgroup)
{
    const uint32_t lbo = kgroup, sbo = 128u;
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// 128-byte-swizzled layouts (what a TMA copy with the 128B swizzle writes):
// rows of 128 bytes (64 bf16), the eight 16-byte chunks of row r stored at
// chunk index c ^ (r % 8), 8-row atoms of 1024 bytes (1024-byte aligned).
// K-major: a row is one M/N index, K runs along the row; the MMA's k-th step
// of 16 elements starts 32 bytes further inside the row, the next 64
// elements of K live in another region of rows.  8-row groups at 1024 bytes.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;                    // leading offset: unused for this layout
    d |= (uint64_t)(1024u >> 4) << 32;          // 8-row group stride
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;                    // 128-byte swizzle
    return d;
}
// MN-major: a row is one K index with 64 consecutive M/N elements; regions of
// 64 M/N elements `region` bytes apart (leading offset), 8-row K groups at
// 1024 bytes (stride offset); the MMA's k-th step of 16 rows starts 2048
// bytes further.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t region)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((region >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, no negation,
// shape M x N (K = 16 per instruction); A K-major; B K-major, or MN-major
// when b_mn_major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn_major = 0)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with A read from tensor memory: row m of A in lane m, two bf16
// per 32-bit column (element 2c in the low half of column c); the k-th step
// of 16 elements starts 8 columns further.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy writes to shared memory become visible to the tensor core.
__device__ __forceinline__ void fence_smem_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Tensor-memory allocation by one whole warp; the base address lands in *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive fp32 columns of this thread's lane (warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31; taddr must carry that lane base).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 8 consecutive 32-bit columns of this thread's lane; completes at the next
// tmem_wait_st().
__device__ __forceinline__ void tmem_st8_async(uint32_t taddr, const uint32_t* r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One poll of phase `parity` (acquire at CTA scope: covers this CTA's own
// writes, the tensor core's commits and transaction bytes that completed on
// the barrier -- including st.async data from a peer CTA).
// The thread may sleep up to kSuspendNs inside one poll (it wakes when the
// phase completes), so waiting warps do not take issue slots from working ones.
constexpr uint32_t kSuspendNs = 2000;
__device__ __forceinline__ bool mbar_test(uint32_t bar_addr, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar_addr), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return done != 0;
}
// Non-blocking test of phase `parity` (never suspends the thread).
__device__ __forceinline__ bool mbar_ready(uint32_t bar_addr, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return done != 0;
}
// Arrive and raise the phase's expected transaction count by `bytes`.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Wait for phase `parity` of `bar` to complete, giving up after max_polls
// polls (each poll may itself suspend briefly).  Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_polls)
{
    const uint32_t a = smem_u32(bar);
    for (uint32_t i = 0; i < max_polls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// ---- TMA row gather and the CTA pair of a cluster ----

// Four rows (row ids r0..r3 of a 2-D tensor map whose box is one row of 64
// bf16 at column x) into 512 contiguous bytes of shared memory, swizzled as
// the map says; the bytes complete on `bar`.  A row id outside the tensor
// (e.g. -1) reads zeros.  x * 2 must be a multiple of 16.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* map, int x, int r0, int r1, int r2, int r3,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}

// The same for 4 bytes, and for 16 bytes given as a uint4.
__device__ __forceinline__ void st_async4(uint32_t remote_addr, float a, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
                 "r"(__float_as_uint(a)), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void st_async16u(uint32_t remote_addr, uint4 v, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

// Bring the 128-byte line at `p` (global memory) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// 16 bytes into another CTA's shared memory; the write completes as
// transaction bytes on that CTA's mbarrier `remote_bar`.
__device__ __forceinline__ void st_async16(uint32_t remote_addr, float a, float b, float c, float d,
                                           uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
                 "r"(remote_bar)
                 : "memory");
}
// Named barrier `id` over `nthreads` threads (a multiple of 32); only where
// every participating thread is certain to arrive.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Per-thread register budget of the executing warpgroup (all four warps execute it).
template <int N>
__device__ __forceinline__ void regs_grow()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_shrink()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
// Every thread of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace skv
