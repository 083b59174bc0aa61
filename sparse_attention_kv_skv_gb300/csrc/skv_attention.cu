// The consumer side of "select, then compute": sparse MLA decode attention
// over the slots an assemble call emitted, read straight from the device hot
// buffer ("SGLang и Tair представили иерархичную Sparse Attention ...",
// paragraph 2: DSA selects the Top-k tokens and computes attention over them
// only), on the tensor cores (tcgen05); plus a self-test of the MMA path.
//
// Per (request, layer) unit: q is [128 heads][576] (MLA: 512-wide latent plus
// 64 rope dims, the same 576 bf16 as a KV row); the keys are the k hot rows
// at slots[0..k) (a -1 slot is masked); scores s = scale * q . key over all
// 576 dims; p = softmax over the keys; out = p . V with V the first 512 dims
// of each key row; lse = log sum exp of the scaled scores.
//
// Kernel layout: persistent clusters of two CTAs (one CTA per SM), each
// cluster walking its share of the units in turn, keys in blocks of 64; blocks
// are numbered across a cluster's units, so the key pipeline and every
// exchange run on from one unit into the next.
// Tensor memory (512 columns of 128 fp32 lanes) holds at most half of the
// 128 x 512 fp32 output, so CTA h owns value dims [256h, 256h + 256) and, to
// split the score product too, score dims [288h, 288h + 288): per block each
// CTA computes a partial S over its 288 dims for all 64 keys.  The scores are
// then finished as a reduce-scatter through distributed shared memory: CTA h
// keeps its partial of keys [32h, 32h + 32), sends the peer its partial of the
// other 32 (st.async, completing on the peer's mbarrier; each value as the
// upper 24 bits of its fp32, relative error at most 2^-16), adds the peer's
// partial of its own keys, and runs the softmax of those 32 keys; the two CTAs
// swap their row maxima (so both take the same block maximum and keep the same
// reference) and their halves of P, so each holds the whole P for O += P V over
// its value half.  Each CTA reads only a 640-byte window of every key row
// (dims [256h, 256h + 320) cover its score and value dims), and no product or
// exponential is computed twice.
//
// Warp roles (512 threads): warpgroup 0 the softmax (thread t <-> head t <->
// tensor-memory lane t; online softmax with a lazily raised reference maximum
// -- the accumulator is rescaled only when a block's maximum exceeds it by
// more than 2^8); warpgroup 1 sends the peer its partial scores; one thread of
// warp 8 issues the MMAs, in whichever of the two streams (S of a later block,
// O += P V of the oldest) is ready first; warps 9-15 gather the key rows of
// each block into a ring of shared-memory stages with TMA (tile::gather4: four
// rows by 64 dims per copy, 128-byte swizzle; a masked slot is an out-of-range
// row, which reads zeros).  Q (this CTA's 288 score dims) sits in tensor memory
// as the A operand of S = Q K^T; the swizzled key stage is both the K-major B
// of S and, read as MN-major, the V of O += P V.  Every wait is bounded: a
// timeout sets the sticky device error bit and the CTA winds down.

#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <string>

#include "skv_ctx.cuh"
#include "tcgen05.cuh"

namespace skv {
namespace {

constexpr int kTcThreads = 128;              // one warpgroup: thread t <-> TMEM lane t <-> row t
constexpr uint32_t kMaxPolls = 1u << 22;     // bound of every spinning mbarrier wait
constexpr uint32_t kMaxSleepPolls = 1u << 20; // bound of a wait whose polls may each sleep (about 2 s)

// D[128][N] = A[128][K] * B^T through shared memory and tensor memory; B is
// [N][K] row-major staged K-major, or (mode bit 0) [K][N] row-major staged
// MN-major; A is staged K-major in shared memory, or (mode bit 1) written to
// tensor memory (row m in lane m) and read from there by the MMA.
__global__ void __launch_bounds__(kTcThreads) mma_selftest_kernel(const uint16_t* __restrict__ A,
                                                                  const uint16_t* __restrict__ B,
                                                                  float* __restrict__ D, int N, int K, int mode,
                                                                  uint32_t* __restrict__ status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool b_mn_major = (mode & 1) != 0, a_tmem = (mode & 2) != 0;
    uint8_t* sA = smem;
    uint8_t* sB = smem + 128 * K * 2;
    const int cpr = K / 8;
    if (!a_tmem) {
        for (int i = tid; i < 128 * cpr; i += kTcThreads) {
            const int r = i / cpr, c = i % cpr;
            *reinterpret_cast<uint4*>(sA + tc::kmajor_chunk_offset(r, c, K)) =
                *reinterpret_cast<const uint4*>(A + (size_t)r * K + c * 8);
        }
    }
    if (!b_mn_major) {
        for (int i = tid; i < N * cpr; i += kTcThreads) {
            const int r = i / cpr, c = i % cpr;
            *reinterpret_cast<uint4*>(sB + tc::kmajor_chunk_offset(r, c, K)) =
                *reinterpret_cast<const uint4*>(B + (size_t)r * K + c * 8);
        }
    } else {  // rows are k, 8-element chunks along n: the K-major layout of a (K x N) tile
        const int cpn = N / 8;
        for (int i = tid; i < K * cpn; i += kTcThreads) {
            const int r = i / cpn, c = i % cpn;
            *reinterpret_cast<uint4*>(sB + tc::kmajor_chunk_offset(r, c, N)) =
                *reinterpret_cast<const uint4*>(B + (size_t)r * N + c * 8);
        }
    }
    uint32_t ncols = 32;
    while ((int)ncols < N) ncols <<= 1;
    if (a_tmem) ncols = 512;  // D in columns [0, N), A in [256, 256 + K / 2)
    if (warp == 0) tc::tmem_alloc(&tmem_base, ncols);
    if (tid == 0) tc::mbar_init(&bar, 1);
    tc::fence_smem_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = tmem_base;
    const uint32_t tlane = taddr + ((uint32_t)(32 * warp) << 16);
    if (a_tmem) {  // thread t writes row t of A: two bf16 per column, in memory order
        const uint32_t* row = reinterpret_cast<const uint32_t*>(A + (size_t)tid * K);
        for (int c0 = 0; c0 < K / 2; c0 += 8) {
            uint32_t w[8];
            for (int j = 0; j < 8; ++j) w[j] = row[c0 + j];
            tc::tmem_st8_async(tlane + 256u + (uint32_t)c0, w);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    if (tid == 0) {
        const uint32_t idesc = tc::idesc_bf16_f32(128, (uint32_t)N, b_mn_major ? 1u : 0u);
        const uint32_t sbo_mn = (uint32_t)N / 8 * 128u;  // 8-k-row group stride of the MN-major B
        for (int s = 0; s < K / 16; ++s) {
            const uint64_t bdesc = b_mn_major ? tc::mnmajor_desc(tc::smem_u32(sB) + 2u * sbo_mn * s, sbo_mn)
                                              : tc::kmajor_desc(tc::smem_u32(sB) + 256u * s, K);
            if (a_tmem)
                tc::mma_bf16_ta(taddr, taddr + 256u + 8u * s, bdesc, idesc, s > 0 ? 1u : 0u);
            else
                tc::mma_bf16(taddr, tc::kmajor_desc(tc::smem_u32(sA) + 256u * s, K), bdesc, idesc, s > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bar);
    }
    const bool ok = tc::mbar_wait(&bar, 0, kMaxPolls);
    tc::fence_after_sync();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            tc::tmem_ld32(tlane + (uint32_t)c0, v);
            for (int j = 0; j < 32 && c0 + j < N; ++j) D[(size_t)tid * N + c0 + j] = v[j];
        }
    } else if (tid == 0) {
        *status = 1u;  // the MMA never signalled completion
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(taddr, ncols);
}

constexpr int kHeads = 128;      // M of every product: one head per tensor-memory lane
constexpr int kDim = 576;        // q / key row length (bf16)
constexpr int kRowBytes = kDim * 2;
constexpr int kVHalf = 256;      // value dims per CTA (of 512)
constexpr int kQKHalf = kDim / 2;                        // score dims per CTA (288)
constexpr int kBlk = 64;         // keys per block (the N of S = Q K^T)
constexpr int kHalfBlk = kBlk / 2;                       // keys of a block whose softmax this CTA finishes
constexpr int kWinBoxes = 5;     // 64-dim column boxes of the key-row window a CTA loads (320 dims)
constexpr int kMaxStages = 4;    // key stages in flight (3 when a long slot list needs the room)
constexpr int kSoftmaxThreads = 128;                     // warpgroup 0: one head a thread
constexpr int kXchgWarp0 = 4;                            // warpgroup 1: sends the peer its partial scores
constexpr int kMmaWarp = 8, kLoadWarp0 = 9, kLoadWarps = 7;
constexpr int kAttnThreads = (kLoadWarp0 + kLoadWarps) * 32;  // 512 (128 registers a thread at launch)
constexpr int kSoftmaxRegs = 192, kXchgRegs = 72, kServiceRegs = 88;  // after the split (see the kernel)
static_assert(128 * (kSoftmaxRegs + kXchgRegs + 2 * kServiceRegs) <= 65536 &&
                  32 * (kSoftmaxRegs + kXchgRegs + 2 * kServiceRegs) <= 16384,
              "the register split must fit the launch's registers, also per SM sub-partition");
constexpr int kGathers = kBlk / 4 * kWinBoxes;           // four-row TMA copies per block (80)
constexpr uint32_t kXBytes = kHeads * kHalfBlk * 3;      // the peer's partial scores of my keys (24-bit): 12288
constexpr int kXChunks = kHalfBlk * 3 / 16;              // 16-byte chunks a head's partial scores take (6)
constexpr uint32_t kPBytes = kHeads * kBlk * 2;          // a P tile, both CTAs' halves (bf16): 16384
constexpr uint32_t kBoxBytes = kBlk * 128;               // one column box of a key stage: 64 rows x 128 B
constexpr uint32_t kStageBytes = kWinBoxes * kBoxBytes;  // 40960
constexpr uint32_t kSmemLimit = 227 * 1024;              // dynamic shared memory a CTA may have (no static part)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320;  // O 256, S 64, Q 144 columns
constexpr float kRescaleLog2 = 8.0f;                     // lazy rescale threshold (factor 256)
static_assert(kColQ + kQKHalf / 2 <= kTmemCols && kColS + kBlk <= kColQ, "tensor-memory columns");

struct alignas(16) AttnCtl;
// Shared-memory layout: the key stages first (1024-byte aligned for the
// swizzle), then the two exchange tiles, the two P tiles and the control
// block.
struct AttnLayout {
    int stages;
    uint32_t off_x, off_p, off_ctl, bytes;
};
__host__ __device__ constexpr uint32_t attend_ctl_bytes();
__host__ __device__ inline AttnLayout attend_layout()
{
    for (int st = kMaxStages;; --st) {
        AttnLayout a{st, (uint32_t)st * kStageBytes, 0, 0, 0};
        a.off_p = a.off_x + 2 * kXBytes;
        a.off_ctl = a.off_p + 2 * kPBytes;
        a.bytes = a.off_ctl + attend_ctl_bytes();
        if (a.bytes <= kSmemLimit || st == 2) return a;
    }
}

// Two floats to a bf16 pair (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t bf2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// 2^x on the special-function unit (approximate, denormal results flush to
// zero; -inf gives 0).  The softmax feeds it x <= 8.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct alignas(16) AttnCtl {
    uint64_t full[kMaxStages];   // key stage landed (TMA transaction bytes; one arrive per loader)
    uint64_t empty[kMaxStages];  // key stage consumed by its last product
    uint64_t s_full;             // partial S of the next block is in tensor memory
    uint64_t s_empty;            // the softmax and exchange warpgroups have read it
    uint64_t adv[2];             // the softmax warpgroup has taken block g's row maxima (adv[g % 2]: a phase
                                 // every second block, so a waiter that falls behind by a block still sees
                                 // its phase -- a parity wait tells only the current and the previous one)
    uint64_t x_full[2];          // the peer's partial scores of my keys of a block have arrived (12288 bytes)
    uint64_t m_full[2];          // the peer's row maxima of a block have arrived (512 bytes)
    uint64_t p_full[2];          // a P tile is complete: my half written, the peer's half arrived (8192 bytes)
    uint64_t pv_done[2];         // O += P V of a block has completed
    uint64_t l_full;             // the peer's share of the softmax denominators has arrived (512 bytes; a phase a unit)
    uint64_t q_ready;            // a unit's Q is in tensor memory (a phase a unit)
    uint64_t o_free;             // the softmax has read a unit's accumulator out of tensor memory (a phase a unit)
    uint64_t fin;                // every MMA this CTA issued has completed
    float mx[2][kHeads];         // [block parity][head] the peer's row maxima of the raw scores
    float lx[kHeads];            // [head] the peer's share of the denominator
    uint32_t tmem_base;
    uint32_t abort;              // a wait of this CTA gave up
};
__host__ __device__ constexpr uint32_t attend_ctl_bytes() { return (uint32_t)sizeof(AttnCtl); }
static_assert(sizeof(AttnCtl) % 16 == 0, "control block alignment");

// Bounded wait on a phase of a local mbarrier, giving up early once the CTA
// has aborted.  (A cluster-scope acquire here would cost several hundred
// cycles per wait; the peer's data arrives as transaction bytes on the local
// barrier, which a CTA-scope acquire observes.)
// The 18 MMAs of S = Q K^T for CTA rank H: step st covers window dims
// e = 32H + 16st, in 64-dim box e / 64 at byte (e % 64) * 2 of the swizzled
// row.  The step's descriptor is the stage's plus that offset in 16-byte units
// (the address field cannot carry: every stage address is below 2^18).
template <int H>
__device__ __forceinline__ void issue_scores(uint32_t tbase, uint64_t dk, uint32_t idesc)
{
#pragma unroll
    for (int st = 0; st < kQKHalf / 16; ++st) {
        constexpr uint32_t e0 = 32u * H;
        const uint32_t e = e0 + 16u * st;
        tc::mma_bf16_ta(tbase + kColS, tbase + kColQ + 8u * st, dk + (((e >> 6) * kBoxBytes + (e & 63u) * 2u) >> 4),
                        idesc, st > 0 ? 1u : 0u);
    }
}

// A partial score crosses the CTA pair as the upper 24 bits of its fp32
// pattern (sign, exponent, 15 mantissa bits), rounded to nearest: relative
// error at most 2^-16, the range of fp32.  Four scores pack into three words.
__device__ __forceinline__ uint32_t f24(float x) { return (__float_as_uint(x) + 0x80u) >> 8; }
__device__ __forceinline__ void pack24(const float* v, uint32_t* w)
{
    const uint32_t a = f24(v[0]), b = f24(v[1]), c = f24(v[2]), d = f24(v[3]);
    w[0] = a | (b << 24);
    w[1] = (b >> 8) | (c << 16);
    w[2] = (c >> 16) | (d << 8);
}
__device__ __forceinline__ void unpack24(const uint32_t* w, float* v)
{
    v[0] = __uint_as_float(w[0] << 8);
    v[1] = __uint_as_float(((w[0] >> 24) | (w[1] << 8)) << 8);
    v[2] = __uint_as_float(((w[1] >> 16) | (w[2] << 16)) << 8);
    v[3] = __uint_as_float(w[2] & 0xFFFFFF00u);
}

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, const volatile uint32_t* abort)
{
    const uint32_t a = tc::smem_u32(bar);
    for (uint32_t i = 0; i < kMaxSleepPolls; ++i) {
        if (tc::mbar_test(a, parity)) return true;
        if ((i & 7u) == 7u && *abort) return false;
    }
    return false;
}

__device__ __forceinline__ void give_up(AttnCtl& c, uint32_t* err)
{
    if (!c.abort) {
        c.abort = 1u;
        atomicOr(err, DEVERR_TIMEOUT);
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
    attend_kernel(const __grid_constant__ CUtensorMap hot_map, Dev d, const int32_t* __restrict__ req_ids,
                  const uint16_t* __restrict__ q, const int32_t* __restrict__ slots, uint16_t* __restrict__ out,
                  float* __restrict__ lse, float scale_log2, AttnLayout lay, int units, int withhold_keys)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    AttnCtl& c = *reinterpret_cast<AttnCtl*>(smem + lay.off_ctl);
    const int nst = lay.stages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;  // this cluster; clusters of the grid
    const uint32_t h = blockIdx.x & 1u, peer = h ^ 1u;     // rank in the cluster = value / score half
    const int k = d.k, S = d.S;
    const int nblk = (k + kBlk - 1) / kBlk;
    // The cluster serves units cl, cl + ncl, ... in order; blocks are numbered across them (g), so the
    // key pipeline, the exchanges and all phase arithmetic run on without a break between units.
    auto req_of = [&](int u, int& b, int& l) -> int32_t {
        b = d.layer_sel >= 0 ? u : u / d.L;
        l = d.layer_sel >= 0 ? d.layer_sel : u % d.L;
        const int32_t r = req_ids[b];
        return r >= 0 && r < d.R ? r : -1;  // not a request: zero output (assemble would have rejected it)
    };
    if (tc::smem_u32(smem) & 1023u) {  // the swizzled key stages need 1024-byte-aligned rows of atoms
        if (tid == 0) atomicOr(&d.ctl[CTL_ERR], DEVERR_TIMEOUT);
        return;  // both CTAs of the cluster see the same layout and leave together
    }
    int gtot = 0;  // blocks of this cluster's real units
    for (int u = cl; u < units; u += ncl) {
        int b, l;
        if (req_of(u, b, l) >= 0) gtot += nblk;
    }
    uint8_t* sK = smem;  // key stages
    uint8_t* sX = smem + lay.off_x;
    uint8_t* sP = smem + lay.off_p;
    volatile uint32_t* abort = &c.abort;

    if (tid == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            tc::mbar_init(&c.full[s], kLoadWarps);
            tc::mbar_init(&c.empty[s], 1);
        }
        tc::mbar_init(&c.s_full, 1);
        tc::mbar_init(&c.s_empty, 2 * kSoftmaxThreads);  // the softmax and the exchange warpgroups
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&c.adv[i], kSoftmaxThreads);
            tc::mbar_init(&c.x_full[i], 1);                // one expect_tx arrival + the peer's bytes
            tc::mbar_init(&c.m_full[i], 1);
            tc::mbar_init(&c.p_full[i], kSoftmaxThreads);  // my half (one of them with expect_tx) + the peer's bytes
            tc::mbar_init(&c.pv_done[i], 1);
        }
        tc::mbar_init(&c.l_full, 1);
        tc::mbar_init(&c.q_ready, kSoftmaxThreads);  // the exchange warpgroup writes Q
        tc::mbar_init(&c.o_free, kSoftmaxThreads);
        tc::mbar_init(&c.fin, 1);
        c.abort = 0u;
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&c.tmem_base, kTmemCols);
    tc::fence_before_sync();
    tc::cluster_sync();  // barriers of both CTAs exist before either sends to the other
    tc::fence_after_sync();
    const uint32_t tbase = c.tmem_base;
    // Register split (warpgroup-wide): softmax 192 a thread, exchange 72, MMA and loaders 88; the
    // shares fit the launch's 512 x 128 in total and on every SM sub-partition (one warp of each
    // warpgroup per sub-partition).
    if (warp >= kMmaWarp) {
        tc::regs_shrink<kServiceRegs>();
        if (warp >= kLoadWarp0) {
            // ---- loaders: seven warps share a block's 80 TMA copies (four key rows x one 64-dim box of
            // this CTA's 320-dim window; a masked slot is row -1, which reads zeros), lane j of warp w
            // issuing copy w + 7j -- TMA issue is paced per issuing thread, so the copies are spread over
            // as many lanes and warps as possible.  The warp fetches a block's 64 slots one block ahead
            // (two a lane) and passes each lane its four rows by shuffle; loader 0 also warms L2 with the
            // rows of the block nst ahead, whose stage frees up last. ----
            const int lw = warp - kLoadWarp0;
            const uint32_t mine = (uint32_t)((kGathers - lw + kLoadWarps - 1) / kLoadWarps);  // copies this loader issues
            int last[kMaxStages] = {-1, -1, -1, -1};  // last block issued into each stage
            bool ok = true;
            int g0 = 0;  // first block of the unit
            // withhold_keys (the timeout self-test only): no copy is ever issued, so the first wait for
            // keys runs out with nothing in flight
            for (int u = cl; ok && !withhold_keys && u < units; u += ncl) {
                int b, l;
                const int32_t r = req_of(u, b, l);
                if (r < 0) continue;
                const int64_t row0 = ((int64_t)r * d.L + l) * S;  // first hot row of this unit
                const int32_t* sl = slots + (size_t)u * k;
                auto fetch = [&](int i, int half) -> int32_t {
                    const int key = i * kBlk + 32 * half + lane;
                    const int32_t slot = key < k ? sl[key] : -1;
                    return slot >= 0 && slot < S ? slot : -1;
                };
                const uint8_t* win = d.hot + (size_t)row0 * kRowBytes + 512u * h;  // this CTA's window of row 0
                int32_t v0 = fetch(0, 0), v1 = fetch(0, 1);
                int32_t w0 = lw == 0 && nst < nblk ? fetch(nst, 0) : -1, w1 = lw == 0 && nst < nblk ? fetch(nst, 1) : -1;
                for (int i = 0; i < nblk; ++i) {
                    const int g = g0 + i, s = g % nst;
                    if (g >= nst && !(ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.empty[s], ((g / nst) - 1) & 1, abort))))
                        break;
                    const int32_t n0 = i + 1 < nblk ? fetch(i + 1, 0) : -1, n1 = i + 1 < nblk ? fetch(i + 1, 1) : -1;
                    if (lane == 0) tc::mbar_arrive_expect_tx(&c.full[s], mine * 512u);
                    __syncwarp();
                    {   // lane j issues copy lw + 7j: one warp instruction for all of this warp's copies
                        const int it = lw + kLoadWarps * lane;
                        const int gr = it / kWinBoxes, cb = it - gr * kWinBoxes;
                        int rr[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int j = (4 * gr + x) & (kBlk - 1);  // key of the block
                            const int32_t a = __shfl_sync(0xFFFFFFFFu, v0, j & 31), b2 = __shfl_sync(0xFFFFFFFFu, v1, j & 31);
                            const int32_t slot = j < 32 ? a : b2;
                            rr[x] = slot >= 0 ? (int)(row0 + slot) : -1;
                        }
                        if ((uint32_t)lane < mine)
                            tc::tma_gather4(tc::smem_u32(sK + s * kStageBytes) + cb * kBoxBytes + gr * 512u, &hot_map,
                                            256 * (int)h + 64 * cb, rr[0], rr[1], rr[2], rr[3], &c.full[s]);
                    }
                    if (lw == 0 && i + nst < nblk) {
#pragma unroll
                        for (int cb = 0; cb < kWinBoxes; ++cb) {
                            if (w0 >= 0) tc::prefetch_l2(win + (size_t)w0 * kRowBytes + 128 * cb);
                            if (w1 >= 0) tc::prefetch_l2(win + (size_t)w1 * kRowBytes + 128 * cb);
                        }
                        const bool more = i + nst + 1 < nblk;
                        w0 = more ? fetch(i + nst + 1, 0) : -1;
                        w1 = more ? fetch(i + nst + 1, 1) : -1;
                    }
                    last[s] = g;
                    v0 = n0;
                    v1 = n1;
                }
                g0 += nblk;
            }
            if (lane == 0) {
                if (!ok) give_up(c, &d.ctl[CTL_ERR]);
                for (int s = 0; s < nst; ++s)  // no copy may still be landing when the CTA leaves
                    if (last[s] >= 0 && !tc::mbar_wait(&c.full[s], (uint32_t)(last[s] / nst) & 1u, kMaxPolls))
                        give_up(c, &d.ctl[CTL_ERR]);
            }
            __syncwarp();
        } else {
            // ---- MMA issuer: whichever product is ready first.  O += P(g) V(g) as soon as P(g) is
            // complete (it frees the key stage for the loaders) and, for a unit's first block, once the
            // softmax has read the previous unit's accumulator; S(g) as soon as its keys have landed,
            // S(g-1) has been read out of tensor memory and its unit's Q is in place.  Both streams are
            // issued in order. ----
            if (lane == 0) {
                const uint32_t idesc_s = tc::idesc_bf16_f32(kHeads, kBlk, 0);
                const uint32_t idesc_o = tc::idesc_bf16_f32(kHeads, kVHalf, 1);
                const uint32_t aK = tc::smem_u32(sK), aP = tc::smem_u32(sP);
                bool ok = true;
                int js = 0, ipv = 0, qn = 0;  // next S block, next P V block, units whose Q is in place
                uint32_t idle = 0;
                while (ok && ipv < gtot) {
                    bool progressed = false;
                    const int pu = ipv / nblk, pi = ipv - pu * nblk;  // unit and block of the next P V
                    if (ipv < js && tc::mbar_ready(tc::smem_u32(&c.p_full[ipv & 1]), (uint32_t)(ipv >> 1) & 1u) &&
                        (pi > 0 || pu == 0 || tc::mbar_ready(tc::smem_u32(&c.o_free), (uint32_t)(pu - 1) & 1u))) {
                        const int bb = ipv & 1, s = ipv % nst;
                        tc::fence_smem_async();  // the peer's half arrived through the generic proxy
                        tc::fence_after_sync();
                        const uint32_t vst = aK + s * kStageBytes;  // value dims are the window's first four boxes
#pragma unroll
                        for (int st = 0; st < kBlk / 16; ++st)
                            tc::mma_bf16(tbase + kColO, tc::kmajor_desc(aP + bb * kPBytes + 256u * st, kBlk),
                                         tc::sw128_mnmajor_desc(vst + 2048u * st, kBoxBytes), idesc_o,
                                         (pi > 0 || st > 0) ? 1u : 0u);
                        tc::mma_commit(&c.pv_done[bb]);
                        tc::mma_commit(&c.empty[s]);
                        ++ipv;
                        progressed = true;
                    }
                    if (js < gtot && js / nblk == qn && tc::mbar_ready(tc::smem_u32(&c.q_ready), (uint32_t)qn & 1u))
                        ++qn;
                    if (js < gtot && js / nblk < qn &&
                        tc::mbar_ready(tc::smem_u32(&c.full[js % nst]), (uint32_t)(js / nst) & 1u) &&
                        (js == 0 || tc::mbar_ready(tc::smem_u32(&c.s_empty), (uint32_t)(js - 1) & 1u))) {
                        const int s = js % nst;
                        tc::fence_after_sync();
                        const uint32_t kst = aK + s * kStageBytes;
                        // fully unrolled per CTA rank, so every step's descriptor is the stage's plus a
                        // constant (the MMA issue rate, not the tensor pipe, bounded this loop)
                        const uint64_t dk = tc::sw128_kmajor_desc(kst);
                        if (h == 0)
                            issue_scores<0>(tbase, dk, idesc_s);
                        else
                            issue_scores<1>(tbase, dk, idesc_s);
                        tc::mma_commit(&c.s_full);
                        ++js;
                        progressed = true;
                    }
                    if (progressed) {
                        idle = 0;
                    } else if (++idle > kMaxPolls || ((idle & 255u) == 0 && *abort)) {
                        ok = false;
                    } else {
                        __nanosleep(32);  // leave issue slots to the warps on this sub-partition
                    }
                }
                if (!ok) give_up(c, &d.ctl[CTL_ERR]);
                tc::mma_commit(&c.fin);
                if (!tc::mbar_wait(&c.fin, 0, kMaxPolls)) give_up(c, &d.ctl[CTL_ERR]);
            }
            __syncwarp();
        }
    } else if (warp >= kXchgWarp0) {
        // ---- exchange warpgroup: thread t <-> head t.  Per unit it first writes the unit's Q into
        // tensor memory (every score product of the previous unit has completed: this warpgroup
        // waited for the last one).  For every block, the peer's 32 keys of my partial S go straight
        // from tensor memory into the peer's exchange tile (st.async; the bytes complete on the
        // peer's x_full).  Block g is sent only once my softmax has taken block g - 2's maxima -- which
        // it cannot do before the peer has read block g - 2's tile, the previous user of the buffer. ----
        tc::regs_shrink<kXchgRegs>();
        const int hd = tid - kSoftmaxThreads;
        const uint32_t tl = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t x_peer = tc::map_to_rank(tc::smem_u32(sX), peer) + (uint32_t)hd * 16u;
        const uint32_t xf0 = tc::map_to_rank(tc::smem_u32(&c.x_full[0]), peer);
        const uint32_t xf1 = tc::map_to_rank(tc::smem_u32(&c.x_full[1]), peer);
        bool ok = true;
        int g0 = 0;
        for (int u = cl; ok && u < units; u += ncl) {
            int b, l;
            if (req_of(u, b, l) < 0) continue;
            {   // Q of the unit: this head's 288 score dims into columns [kColQ, kColQ + 144)
                const uint4* qr = reinterpret_cast<const uint4*>(q + ((size_t)u * kHeads + hd) * kDim + h * kQKHalf);
#pragma unroll 3
                for (int gq = 0; gq < kQKHalf / 32; ++gq) {  // 9 groups of 16 columns
                    uint4 a = qr[4 * gq], bq = qr[4 * gq + 1], cq4 = qr[4 * gq + 2], dq = qr[4 * gq + 3];
                    const uint32_t w0[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
                    const uint32_t w1[8] = {cq4.x, cq4.y, cq4.z, cq4.w, dq.x, dq.y, dq.z, dq.w};
                    tc::tmem_st8_async(tl + kColQ + 16u * gq, w0);
                    tc::tmem_st8_async(tl + kColQ + 16u * gq + 8u, w1);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                tc::mbar_arrive(&c.q_ready);
            }
            for (int i = 0; ok && i < nblk; ++i) {
                const int g = g0 + i;
                // warm L2 with the next unit's Q row a few blocks before it is loaded (earlier, the key rows
                // streaming through L2 in the meantime would evict it)
                if (i == (nblk > 3 ? nblk - 3 : 0) && u + ncl < units) {
                    const uint8_t* nq = reinterpret_cast<const uint8_t*>(q + ((size_t)(u + ncl) * kHeads + hd) * kDim + h * kQKHalf);
#pragma unroll
                    for (int x = 0; x < 5; ++x) tc::prefetch_l2(nq + 128 * x);
                }
                if (g >= 2 && !(ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.adv[g & 1], (uint32_t)((g - 2) >> 1) & 1u, abort))))
                    break;
                if (!(ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.s_full, (uint32_t)g & 1u, abort)))) break;
                tc::fence_after_sync();
                float v[kHalfBlk];
                tc::tmem_ld32(tl + kColS + (uint32_t)(kHalfBlk * peer), v);
                tc::fence_before_sync();
                tc::mbar_arrive(&c.s_empty);
                const uint32_t xb = x_peer + (uint32_t)(g & 1) * kXBytes;
                const uint32_t rb = (g & 1) ? xf1 : xf0;
                uint32_t w[kXChunks * 4];
#pragma unroll
                for (int j = 0; j < kHalfBlk / 4; ++j) pack24(v + 4 * j, w + 3 * j);
#pragma unroll
                for (int m = 0; m < kXChunks; ++m)
                    tc::st_async16u(xb + 2048u * m, make_uint4(w[4 * m], w[4 * m + 1], w[4 * m + 2], w[4 * m + 3]), rb);
            }
            g0 += nblk;
        }
        if (!ok) give_up(c, &d.ctl[CTL_ERR]);
    } else {
        // ---- softmax warpgroup: thread t <-> head t <-> tensor-memory lane t, my 32 keys of every
        // block (keys [32h, 32h + 32)); both CTAs take the same block maxima, so they keep the same
        // reference and their P halves fit one P V product ----
        tc::regs_grow<kSoftmaxRegs>();
        const int hd = tid;
        const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
        const uint32_t mx_peer = tc::map_to_rank(tc::smem_u32(&c.mx[0][0]), peer) + (uint32_t)hd * 4u;
        const uint32_t mf0 = tc::map_to_rank(tc::smem_u32(&c.m_full[0]), peer);
        const uint32_t mf1 = tc::map_to_rank(tc::smem_u32(&c.m_full[1]), peer);
        const uint32_t p_peer = tc::map_to_rank(tc::smem_u32(sP), peer);
        const uint32_t pf0 = tc::map_to_rank(tc::smem_u32(&c.p_full[0]), peer);
        const uint32_t pf1 = tc::map_to_rank(tc::smem_u32(&c.p_full[1]), peer);
        const uint32_t lx_peer = tc::map_to_rank(tc::smem_u32(&c.lx[0]), peer) + (uint32_t)hd * 4u;
        const uint32_t lf_peer = tc::map_to_rank(tc::smem_u32(&c.l_full), peer);
        auto own = [&](int j, float (&dst)[kHalfBlk]) -> bool {  // my keys of my partial S(j)
            if (!__all_sync(0xFFFFFFFFu, wait_phase(&c.s_full, (uint32_t)j & 1u, abort))) return false;
            tc::fence_after_sync();
            tc::tmem_ld32(tl + kColS + (uint32_t)(kHalfBlk * h), dst);
            tc::fence_before_sync();
            tc::mbar_arrive(&c.s_empty);
            return true;
        };
        float cur[kHalfBlk];  // my partial S of the block being processed, my keys
        bool ok = true;
        if (gtot > 0) {
            if (tid == 0) tc::mbar_arrive_expect_tx(&c.x_full[0], kXBytes);
            ok = own(0, cur);
        }
        int g0 = 0, n = 0;  // first block of the unit; units done
        for (int u = cl; u < units; u += ncl) {
            int b, l;
            if (req_of(u, b, l) < 0) {  // not a request: zeros and lse = -inf, nothing else takes part
                uint16_t* o = out + ((size_t)u * kHeads + hd) * 512 + h * kVHalf;
                for (int cc = 0; cc < kVHalf; cc += 8) *reinterpret_cast<uint4*>(o + cc) = make_uint4(0, 0, 0, 0);
                if (h == 0 && lse) lse[(size_t)u * kHeads + hd] = -INFINITY;
                continue;
            }
            if (!ok) continue;
            const int32_t* sl = slots + (size_t)u * k;
            auto slot_of = [&](int i) -> int32_t {  // the slot of my key `lane` of block i
                const int key = i * kBlk + kHalfBlk * (int)h + lane;
                return key < k ? sl[key] : -1;
            };
            float m_ref = -INFINITY;  // reference maximum (log2 domain) the exponentials use; equal in both CTAs
            float l_run = 0.0f;       // this CTA's share of the softmax denominator
            int32_t sp = slot_of(0);
            for (int i = 0; ok && i < nblk; ++i) {
                const int g = g0 + i, bb = g & 1;
                const uint32_t ph = (uint32_t)(g >> 1) & 1u;
                if (!(ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.x_full[bb], ph, abort)))) break;
                float sv[kHalfBlk];  // mine + the peer's partial: the full scores of my keys
                const uint8_t* xrow = sX + bb * kXBytes + hd * 16;
                uint32_t xw[kXChunks * 4];
#pragma unroll
                for (int m = 0; m < kXChunks; ++m) {
                    const uint4 pr = *reinterpret_cast<const uint4*>(xrow + 2048 * m);
                    xw[4 * m] = pr.x;
                    xw[4 * m + 1] = pr.y;
                    xw[4 * m + 2] = pr.z;
                    xw[4 * m + 3] = pr.w;
                }
#pragma unroll
                for (int j = 0; j < kHalfBlk / 4; ++j) {
                    float px[4];
                    unpack24(xw + 3 * j, px);
#pragma unroll
                    for (int e = 0; e < 4; ++e) sv[4 * j + e] = cur[4 * j + e] + px[e];
                }
                const int32_t sp_next = i + 1 < nblk ? slot_of(i + 1) : -1;  // in flight while this block runs
                if (g + 1 < gtot && tid == 0) tc::mbar_arrive_expect_tx(&c.x_full[bb ^ 1], kXBytes);
                const uint32_t vm = __ballot_sync(0xFFFFFFFFu, sp >= 0 && sp < S);
                if (vm != 0xFFFFFFFFu) {
#pragma unroll
                    for (int j = 0; j < kHalfBlk; ++j) sv[j] = (vm >> j) & 1u ? sv[j] : -INFINITY;
                }
                float mx[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mx[j] = fmaxf(fmaxf(fmaxf(sv[j], sv[j + 4]), fmaxf(sv[j + 8], sv[j + 12])),
                                  fmaxf(fmaxf(sv[j + 16], sv[j + 20]), fmaxf(sv[j + 24], sv[j + 28])));
                const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                // P tile bb (mine and, once I send my maxima, the peer's half) is free once O += P(g-2)
                // V(g-2) has completed; the peer sends its P(g) only after my maxima of block g
                if (g >= 2 && !(ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.pv_done[bb], ((g - 2) >> 1) & 1, abort))))
                    break;
                if (tid == 0) tc::mbar_arrive_expect_tx(&c.m_full[bb], kHeads * 4u);
                tc::st_async4(mx_peer + (uint32_t)bb * kHeads * 4u, mloc, bb ? mf1 : mf0);
                if (!(ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.m_full[bb], ph, abort)))) break;
                const float mb = fmaxf(mloc, c.mx[bb][hd]) * scale_log2;  // the same in both CTAs
                tc::mbar_arrive(&c.adv[bb]);  // the exchange warpgroup may now send block g + 2
                float factor = 1.0f;
                if (mb > m_ref + kRescaleLog2) {
                    factor = m_ref == -INFINITY ? 0.0f : ex2(m_ref - mb);
                    m_ref = mb;
                    l_run *= factor;
                }
                if (i > 0 && __any_sync(0xFFFFFFFFu, factor != 1.0f)) {  // rescale this warp's rows of O
                    if (!(ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort))))
                        break;
                    tc::fence_after_sync();
                    for (int c0 = 0; c0 < kVHalf; c0 += 32) {
                        float ov[32];
                        tc::tmem_ld32(tl + kColO + c0, ov);
#pragma unroll
                        for (int j = 0; j < 32; ++j) ov[j] *= factor;
                        tc::tmem_st32(tl + kColO + c0, ov);
                    }
                    tc::fence_before_sync();
                }
                // p = 2^(s * scale - m_ref); masked keys give 2^-inf = 0.  While no
                // real key has been seen (m_ref = -inf for every head) all p are 0.
                uint32_t pk[kHalfBlk / 2];
                float ps[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (m_ref != -INFINITY) {
                    const float neg_m = -m_ref;
#pragma unroll
                    for (int j = 0; j < kHalfBlk; j += 2) {
                        const float p0 = ex2(fmaf(sv[j], scale_log2, neg_m));
                        const float p1 = ex2(fmaf(sv[j + 1], scale_log2, neg_m));
                        ps[(j >> 1) & 3] += p0 + p1;
                        pk[j / 2] = bf2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kHalfBlk / 2; ++j) pk[j] = 0u;
                }
                l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
                // my half of P(g): into my tile and into the peer's, at the same place (keys [32h, 32h + 32))
                const uint32_t pb = (uint32_t)bb * kPBytes;
#pragma unroll
                for (int cc = 0; cc < kHalfBlk / 8; ++cc) {
                    const uint32_t off = pb + tc::kmajor_chunk_offset(hd, 4 * h + cc, kBlk);
                    const uint4 w4 = make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                    *reinterpret_cast<uint4*>(sP + off) = w4;
                    tc::st_async16u(p_peer + off, w4, bb ? pf1 : pf0);
                }
                tc::fence_smem_async();
                if (tid == 0)
                    tc::mbar_arrive_expect_tx(&c.p_full[bb], kPBytes / 2);  // my arrival + the peer's half
                else
                    tc::mbar_arrive(&c.p_full[bb]);
                sp = sp_next;
                // S of the next block of this unit, read once P(g) is out: its product ran while this
                // block's softmax did, and the product after it is issued behind O += P(g) V(g), so it
                // does not delay the release of this block's key stage.  The next unit's first S waits
                // for that unit's Q, so it is read after this unit's epilogue instead.
                if (g + 1 < gtot && i + 1 < nblk && !(ok = own(g + 1, cur))) break;
            }
            const int gl = g0 + nblk - 1;  // the unit's last block
            // the denominator: CTA 0's share + CTA 1's share, in that order on both CTAs (sent
            // before waiting for the last O += P V, so the two waits overlap)
            if (tid == 0) tc::mbar_arrive_expect_tx(&c.l_full, kHeads * 4u);
            tc::st_async4(lx_peer, l_run, lf_peer);
            if (ok) ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.pv_done[gl & 1], ((gl >> 1) & 1), abort));
            if (ok) ok = __all_sync(0xFFFFFFFFu, wait_phase(&c.l_full, (uint32_t)n & 1u, abort));
            if (ok) {
                const float l_all = h == 0 ? l_run + c.lx[hd] : c.lx[hd] + l_run;
                tc::fence_after_sync();
                const float inv = l_all > 0.0f ? 1.0f / l_all : 0.0f;
                // O goes out through shared memory so that every store instruction writes whole rows:
                // thread hd puts its row (this CTA's 256 value dims as bf16) into a staging area, 128
                // columns at a time; then the warp stores its 32 rows two at a time, 16 lanes a row.
                // The staging area of warp w is its 4 KB of each P tile (rows 0-15 in tile 0, 16-31 in
                // tile 1): bytes no other thread writes before this warp's next P write, since O += P V
                // of this unit has completed and the peer writes a P tile only after every thread here
                // has sent it the next block's maxima.  16-byte chunk c of staged row r sits at chunk
                // position c ^ (r % 16), which keeps both passes free of bank conflicts.
                uint8_t* stage = sP + 4096u * (uint32_t)warp;
                uint16_t* orow = out + ((size_t)u * kHeads + (hd & ~31)) * 512 + h * kVHalf;  // the warp's first row
                uint8_t* mine = stage + (lane >> 4) * kPBytes + (lane & 15) * 256;
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int c0 = 0; c0 < 128; c0 += 32) {
                        float ov[32];
                        tc::tmem_ld32(tl + kColO + (uint32_t)(half * 128 + c0), ov);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(mine + (((c0 / 8 + q) ^ (lane & 15)) << 4)) =
                                make_uint4(bf2(ov[8 * q] * inv, ov[8 * q + 1] * inv), bf2(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv),
                                           bf2(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv), bf2(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv));
                    }
                    __syncwarp();
#pragma unroll 4
                    for (int i = 0; i < 16; ++i) {
                        const int r = 2 * i + (lane >> 4), cc = lane & 15;
                        const uint4 w = *reinterpret_cast<const uint4*>(stage + (r >> 4) * kPBytes + (r & 15) * 256 +
                                                                        ((cc ^ (r & 15)) << 4));
                        *reinterpret_cast<uint4*>(orow + (size_t)r * 512 + half * 128 + cc * 8) = w;
                    }
                    __syncwarp();
                }
                if (h == 0 && lse)
                    lse[(size_t)u * kHeads + hd] = l_all > 0.0f ? (m_ref + log2f(l_all)) * 0.69314718055994531f : -INFINITY;
                tc::fence_before_sync();
                tc::mbar_arrive(&c.o_free);  // the next unit's first O += P V may overwrite the accumulator
            }
            if (ok && gl + 1 < gtot) ok = own(gl + 1, cur);  // the first S of the next unit
            g0 += nblk;
            ++n;
        }
        if (!ok) give_up(c, &d.ctl[CTL_ERR]);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync();  // neither CTA leaves while the other may still write into its shared memory
    if (tid == 0 && *abort) {
        // A wait of this CTA gave up, so bytes the peer sent before it arrived at the cluster
        // barrier may still be landing here (nothing waited for them): keep the shared memory
        // allocated a while longer.
        for (int i = 0; i < 64; ++i) __nanosleep(1000);
    }
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

size_t attend_smem_bytes(int) { return attend_layout().bytes; }

// The hot buffer as a 2-D tensor of R*L*S rows by 576 bf16 (row stride 1152
// bytes) for TMA: box one row by 64 columns, 128-byte swizzle, out-of-range
// rows read as zeros.  cuTensorMapEncodeTiled is reached through the runtime's
// driver entry point (no link against the driver library).
cudaError_t encode_hot_map(const Dev& d, CUtensorMap* map)
{
    const uint64_t rows = (uint64_t)d.R * (uint64_t)d.L * (uint64_t)d.S;
    if (rows > 0x7FFFFFFFull || d.row_bytes != kRowBytes) return cudaErrorInvalidValue;
    using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static EncodeTiled encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult found = cudaDriverEntryPointSymbolNotFound;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                               &found);
        if (e != cudaSuccess) return e;
        if (found != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = reinterpret_cast<EncodeTiled>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kRowBytes};
    const cuuint32_t box[2] = {64, 1}, elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d.hot, dims, strides, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t prepare_attend(int* device_sms)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(device_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)  // a function attribute is per device: set on the device the context lives on
        e = cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
    return e;
}

cudaError_t launch_attend(const void* hot_map, const Dev& d, const int32_t* req_ids, int B, const void* q,
                          const int32_t* slots, void* out, float* lse, float sm_scale, int max_sms, int device_sms,
                          cudaStream_t st, bool withhold_keys)
{
    const AttnLayout lay = attend_layout();
    if (d.k > (int)kMaxTopk || lay.bytes > kSmemLimit || device_sms < 2) return cudaErrorInvalidValue;
    // a persistent grid: one cluster per two SMs (one CTA per SM), at most one per unit
    const int units = call_units(d, B);
    const int use_sms = max_sms > 0 ? std::min(max_sms, device_sms) : device_sms;
    const int clusters = std::max(1, std::min(units, use_sms / 2));
    attend_kernel<<<clusters * 2, kAttnThreads, lay.bytes, st>>>(
        *static_cast<const CUtensorMap*>(hot_map), d, req_ids, static_cast<const uint16_t*>(q), slots,
        static_cast<uint16_t*>(out), lse, sm_scale * 1.4426950408889634f, lay, units, withhold_keys ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace skv

namespace {
skv_status attend_impl(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B, int32_t layer, const void* q_dev,
                       const int32_t* slots_dev, void* out_dev, float* lse_dev, float sm_scale, skv_stream_t stream,
                       bool withhold_keys, const char* what)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch || layer < -1 || layer >= ctx->cfg.num_layers ||
        !(sm_scale > 0.0f) || !std::isfinite(sm_scale))
        return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids_dev || !q_dev || !slots_dev || !out_dev || ctx->cfg.row_bytes != skv::kDim * 2)
        return SKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(out_dev)) & 15u) return SKV_ERR_INVALID_ARG;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != ctx->cfg.device && cudaSetDevice(ctx->cfg.device) != cudaSuccess) return SKV_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (!ctx->hot_map_ready) {  // host-side encoding only: safe while a stream is being captured
        e = skv::encode_hot_map(ctx->d, &ctx->hot_map);
        ctx->hot_map_ready = e == cudaSuccess;
    }
    skv::Dev d = ctx->d;
    d.layer_sel = layer;
    if (e == cudaSuccess)
        e = skv::launch_attend(&ctx->hot_map, d, req_ids_dev, B, q_dev, slots_dev, out_dev, lse_dev, sm_scale,
                               ctx->attend_sms, ctx->device_sms, stream, withhold_keys);
    if (prev >= 0 && prev != ctx->cfg.device) cudaSetDevice(prev);
    if (e != cudaSuccess) {
        skv::set_last_error_message((std::string(what) + ": " + cudaGetErrorString(e)).c_str());
        return SKV_ERR_CUDA;
    }
    return SKV_OK;
}
}  // namespace

extern "C" skv_status skv_attend(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B, int32_t layer, const void* q_dev,
                                 const int32_t* slots_dev, void* out_dev, float* lse_dev, float sm_scale,
                                 skv_stream_t stream)
{
    return attend_impl(ctx, req_ids_dev, B, layer, q_dev, slots_dev, out_dev, lse_dev, sm_scale, stream, false,
                       "skv_attend");
}

extern "C" skv_status skv_selftest_attend_timeout(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B,
                                                  const void* q_dev, const int32_t* slots_dev, void* out_dev,
                                                  skv_stream_t stream)
{
    return attend_impl(ctx, req_ids_dev, B, -1, q_dev, slots_dev, out_dev, nullptr, 1.0f, stream, true,
                       "skv_selftest_attend_timeout");
}

extern "C" skv_status skv_set_attend_sms(skv_ctx* ctx, int32_t sms)
{
    if (!ctx || sms < 0) return SKV_ERR_INVALID_ARG;
    ctx->attend_sms = sms;
    return SKV_OK;
}

extern "C" skv_status skv_selftest_mma(const void* a_dev, const void* b_dev, float* d_dev, int32_t n, int32_t k,
                                       int32_t mode, skv_stream_t stream)
{
    if (!a_dev || !b_dev || !d_dev || n < 16 || n > 256 || n % 16 || k < 16 || k > 128 || k % 16 || mode < 0 ||
        mode > 3)
        return SKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a_dev) | reinterpret_cast<uintptr_t>(b_dev)) & 15u) return SKV_ERR_INVALID_ARG;
    uint32_t* status = nullptr;
    cudaError_t e = cudaMallocAsync(&status, 4, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, 4, stream);
    const int smem = 128 * k * 2 + n * k * 2;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(skv::mma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) {
        skv::mma_selftest_kernel<<<1, skv::kTcThreads, smem, stream>>>(static_cast<const uint16_t*>(a_dev),
                                                                        static_cast<const uint16_t*>(b_dev), d_dev,
                                                                        n, k, mode, status);
        e = cudaGetLastError();
    }
    uint32_t h = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, status, 4, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (status) cudaFreeAsync(status, stream);
    if (e != cudaSuccess) {
        skv::set_last_error_message((std::string("skv_selftest_mma: ") + cudaGetErrorString(e)).c_str());
        return SKV_ERR_CUDA;
    }
    if (h) {
        skv::set_last_error_message("skv_selftest_mma: the tensor-core MMA did not complete in time");
        return SKV_ERR_CUDA;
    }
    return SKV_OK;
}
