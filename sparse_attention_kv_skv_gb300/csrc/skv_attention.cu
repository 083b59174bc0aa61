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
// Kernel layout: two CTAs per unit, one per half of the 512 value dims (the
// fp32 output of 128 heads x 512 dims would fill all of tensor memory); 128
// threads, thread t <-> head t <-> tensor-memory lane t.  Q stays in shared
// memory for the whole unit; keys stream in blocks of 32: S = Q K^T (M 128,
// N 32, K 576) into tensor memory, an online softmax per head (the reference
// maximum is raised, and the accumulator rescaled, only when a block's maximum
// exceeds it by more than 2^8, so rescales are rare), P (bf16) to shared
// memory, O += P V (M 128, N 256, K 32) with V read in place from the key
// block as an MN-major operand.  The next block's rows are loaded into
// registers while the current block's products run.

#include <cuda_bf16.h>

#include <cmath>
#include <string>

#include "skv_ctx.cuh"
#include "tcgen05.cuh"

namespace skv {
namespace {

constexpr int kTcThreads = 128;              // one warpgroup: thread t <-> TMEM lane t <-> row t
constexpr uint32_t kMaxPolls = 1u << 22;     // bound of every mbarrier wait

// D[128][N] = A[128][K] * B^T through shared memory and tensor memory; B is
// [N][K] row-major staged K-major, or (b_mn_major) [K][N] row-major staged
// MN-major.
__global__ void __launch_bounds__(kTcThreads) mma_selftest_kernel(const uint16_t* __restrict__ A,
                                                                  const uint16_t* __restrict__ B,
                                                                  float* __restrict__ D, int N, int K,
                                                                  int b_mn_major, uint32_t* __restrict__ status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5;
    uint8_t* sA = smem;
    uint8_t* sB = smem + 128 * K * 2;
    const int cpr = K / 8;
    for (int i = tid; i < 128 * cpr; i += kTcThreads) {
        const int r = i / cpr, c = i % cpr;
        *reinterpret_cast<uint4*>(sA + tc::kmajor_chunk_offset(r, c, K)) =
            *reinterpret_cast<const uint4*>(A + (size_t)r * K + c * 8);
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
    if (warp == 0) tc::tmem_alloc(&tmem_base, ncols);
    if (tid == 0) tc::mbar_init(&bar, 1);
    tc::fence_smem_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = tmem_base;
    if (tid == 0) {
        const uint32_t idesc = tc::idesc_bf16_f32(128, (uint32_t)N, b_mn_major ? 1u : 0u);
        const uint32_t sbo_mn = (uint32_t)N / 8 * 128u;  // 8-k-row group stride of the MN-major B
        for (int s = 0; s < K / 16; ++s) {
            const uint64_t bdesc = b_mn_major ? tc::mnmajor_desc(tc::smem_u32(sB) + 2u * sbo_mn * s, sbo_mn)
                                              : tc::kmajor_desc(tc::smem_u32(sB) + 256u * s, K);
            tc::mma_bf16(taddr, tc::kmajor_desc(tc::smem_u32(sA) + 256u * s, K), bdesc, idesc, s > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bar);
    }
    const bool ok = tc::mbar_wait(&bar, 0, kMaxPolls);
    tc::fence_after_sync();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            tc::tmem_ld32(taddr + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
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
constexpr int kVHalf = 256;      // value dims per CTA (of 512)
constexpr int kBlk = 32;         // keys per block
constexpr int kChunks = kDim / 8;                       // 16-byte chunks per row (72)
constexpr int kPre = kBlk * kChunks / kTcThreads;       // prefetched chunks per thread (18)
constexpr uint32_t kSmemQ = kHeads * kDim * 2;          // 147456
constexpr uint32_t kSmemK = kBlk * kDim * 2;            // 36864
constexpr uint32_t kSmemP = kHeads * kBlk * 2;          // 8192
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;              // S: 32 columns, O: 256 columns
constexpr float kRescaleLog2 = 8.0f;                    // lazy rescale threshold (factor 256)

__device__ __forceinline__ uint16_t f2bf(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// Rows of key block starting at j0 into registers: chunk i of this thread is
// chunk (tid + i * 128) of the block, row j = that / 72.  Masked or
// out-of-range slots give zero rows.
__device__ __forceinline__ void load_block(uint4 (&pre)[kPre], const uint8_t* hot_u, const int32_t* sl, int k, int S,
                                           int j0, int tid)
{
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
        const int ci = tid + i * kTcThreads;
        const int j = ci / kChunks, c = ci - j * kChunks;
        const int key = j0 + j;
        const int32_t slot = key < k ? sl[key] : -1;
        pre[i] = (slot >= 0 && slot < S)
                     ? *reinterpret_cast<const uint4*>(hot_u + (size_t)slot * (kDim * 2) + c * 16)
                     : make_uint4(0, 0, 0, 0);
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) attend_kernel(Dev d, const int32_t* __restrict__ req_ids,
                                                               const uint16_t* __restrict__ q,
                                                               const int32_t* __restrict__ slots,
                                                               uint16_t* __restrict__ out, float* __restrict__ lse,
                                                               float scale_log2)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int32_t valid[kBlk];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int uc = blockIdx.x >> 1, vh = blockIdx.x & 1;  // unit of the call, value half
    const int b = d.layer_sel >= 0 ? uc : uc / d.L;
    const int l = d.layer_sel >= 0 ? d.layer_sel : uc % d.L;
    const int32_t r = req_ids[b];
    const int k = d.k, S = d.S;
    uint16_t* out_u = out + ((size_t)uc * kHeads + tid) * 512 + vh * kVHalf;
    if (r < 0 || r >= d.R) {  // not a request: zero output (assemble would have rejected it)
        for (int c = 0; c < kVHalf; c += 8) *reinterpret_cast<uint4*>(out_u + c) = make_uint4(0, 0, 0, 0);
        if (vh == 0 && lse) lse[(size_t)uc * kHeads + tid] = -INFINITY;
        return;
    }
    const uint8_t* hot_u = d.hot + (size_t)((int64_t)r * d.L + l) * S * (kDim * 2);
    const int32_t* sl = slots + (size_t)uc * k;
    uint8_t* sQ = smem;
    uint8_t* sK = smem + kSmemQ;
    uint8_t* sP = sK + kSmemK;

    // Q of this unit, K-major
    const uint16_t* q_u = q + (size_t)uc * kHeads * kDim;
    for (int i = tid; i < kHeads * kChunks; i += kTcThreads) {
        const int h = i / kChunks, c = i - h * kChunks;
        *reinterpret_cast<uint4*>(sQ + tc::kmajor_chunk_offset(h, c, kDim)) =
            *reinterpret_cast<const uint4*>(q_u + (size_t)h * kDim + c * 8);
    }
    if (warp == 0) tc::tmem_alloc(&tmem_base, kTmemCols);
    if (tid == 0) tc::mbar_init(&bar, 1);
    uint4 pre[kPre];
    load_block(pre, hot_u, sl, k, S, 0, tid);
    tc::fence_smem_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tmem_base;
    const uint32_t tlane = tbase + ((uint32_t)(32 * warp) << 16);
    const uint32_t idesc_s = tc::idesc_bf16_f32(kHeads, kBlk, 0);
    const uint32_t idesc_o = tc::idesc_bf16_f32(kHeads, kVHalf, 1);
    const uint32_t aQ = tc::smem_u32(sQ), aK = tc::smem_u32(sK), aP = tc::smem_u32(sP);
    const uint32_t kgroup = kDim / 8 * 128;  // 8-key group stride of the key block (9216 B)

    float m_ref = -INFINITY;  // reference maximum (log2 domain) the exponentials use
    float l_run = 0.0f;
    uint32_t phase = 0;
    bool ok = true;
    const int nblk = (k + kBlk - 1) / kBlk;
    for (int blk = 0; blk < nblk && ok; ++blk) {
        const int j0 = blk * kBlk;
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            const int ci = tid + i * kTcThreads;
            const int j = ci / kChunks, c = ci - j * kChunks;
            *reinterpret_cast<uint4*>(sK + tc::kmajor_chunk_offset(j, c, kDim)) = pre[i];
        }
        if (tid < kBlk) {
            const int key = j0 + tid;
            const int32_t slot = key < k ? sl[key] : -1;
            valid[tid] = slot >= 0 && slot < S;
        }
        tc::fence_smem_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (blk + 1 < nblk) load_block(pre, hot_u, sl, k, S, j0 + kBlk, tid);  // in flight during the products

        // S = Q K^T
        if (tid == 0) {
            for (int s = 0; s < kDim / 16; ++s)
                tc::mma_bf16(tbase + kColS, tc::kmajor_desc(aQ + 256u * s, kDim), tc::kmajor_desc(aK + 256u * s, kDim),
                             idesc_s, s > 0 ? 1u : 0u);
            tc::mma_commit(&bar);
        }
        ok = __syncthreads_and(tc::mbar_wait(&bar, phase, kMaxPolls));  // one decision for the whole CTA
        phase ^= 1u;
        tc::fence_after_sync();
        if (!ok) break;
        float sv[32];
        tc::tmem_ld32(tlane + kColS, sv);

        // online softmax of this head over the block
        float mb = -INFINITY;
#pragma unroll
        for (int j = 0; j < kBlk; ++j) {
            sv[j] = valid[j] ? sv[j] * scale_log2 : -INFINITY;
            mb = fmaxf(mb, sv[j]);
        }
        float factor = 1.0f;
        if (mb > m_ref + kRescaleLog2) {
            factor = m_ref == -INFINITY ? 0.0f : exp2f(m_ref - mb);
            m_ref = mb;
            l_run *= factor;
        }
        if (blk > 0 && __any_sync(0xFFFFFFFFu, factor != 1.0f)) {  // rescale this warp's rows of O
            for (int c0 = 0; c0 < kVHalf; c0 += 32) {
                float ov[32];
                tc::tmem_ld32(tlane + kColO + c0, ov);
#pragma unroll
                for (int j = 0; j < 32; ++j) ov[j] *= factor;
                tc::tmem_st32(tlane + kColO + c0, ov);
            }
        }
        float psum = 0.0f;
        uint32_t pk[kBlk / 2];
#pragma unroll
        for (int j = 0; j < kBlk; j += 2) {
            const float p0 = sv[j] == -INFINITY ? 0.0f : exp2f(sv[j] - m_ref);
            const float p1 = sv[j + 1] == -INFINITY ? 0.0f : exp2f(sv[j + 1] - m_ref);
            psum += p0 + p1;
            pk[j / 2] = (uint32_t)f2bf(p0) | ((uint32_t)f2bf(p1) << 16);
        }
        l_run += psum;
#pragma unroll
        for (int c = 0; c < kBlk / 8; ++c)
            *reinterpret_cast<uint4*>(sP + tc::kmajor_chunk_offset(tid, c, kBlk)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        tc::fence_smem_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();

        // O += P V, V = dims [vh*256, vh*256 + 256) of the key block, MN-major
        if (tid == 0) {
            for (int s = 0; s < kBlk / 16; ++s)
                tc::mma_bf16(tbase + kColO, tc::kmajor_desc(aP + 256u * s, kBlk),
                             tc::mnmajor_desc(aK + (uint32_t)vh * (kVHalf / 8) * 128u + 2u * kgroup * s, kgroup),
                             idesc_o, (blk > 0 || s > 0) ? 1u : 0u);
            tc::mma_commit(&bar);
        }
        ok = __syncthreads_and(tc::mbar_wait(&bar, phase, kMaxPolls));
        phase ^= 1u;
        tc::fence_after_sync();
    }

    if (ok) {
        const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
        for (int c0 = 0; c0 < kVHalf; c0 += 32) {
            float ov[32];
            tc::tmem_ld32(tlane + kColO + c0, ov);
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) w[j / 2] = (uint32_t)f2bf(ov[j] * inv) | ((uint32_t)f2bf(ov[j + 1] * inv) << 16);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(out_u + c0 + 8 * c) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
        if (vh == 0 && lse)
            lse[(size_t)uc * kHeads + tid] = l_run > 0.0f ? (m_ref + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    } else if (tid == 0) {
        atomicOr(&d.ctl[CTL_ERR], DEVERR_TIMEOUT);  // a product never signalled completion
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

size_t attend_smem_bytes() { return kSmemQ + kSmemK + kSmemP; }

cudaError_t launch_attend(const Dev& d, const int32_t* req_ids, int B, const void* q, const int32_t* slots,
                          void* out, float* lse, float sm_scale, cudaStream_t st)
{
    static const size_t smem = attend_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_kernel<<<call_units(d, B) * 2, kTcThreads, smem, st>>>(d, req_ids, static_cast<const uint16_t*>(q), slots,
                                                                   static_cast<uint16_t*>(out), lse,
                                                                   sm_scale * 1.4426950408889634f);
    return cudaGetLastError();
}

}  // namespace skv

extern "C" skv_status skv_attend(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B, int32_t layer, const void* q_dev,
                                 const int32_t* slots_dev, void* out_dev, float* lse_dev, float sm_scale,
                                 skv_stream_t stream)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch || layer < -1 || layer >= ctx->cfg.num_layers)
        return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids_dev || !q_dev || !slots_dev || !out_dev || ctx->cfg.row_bytes != skv::kDim * 2)
        return SKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(out_dev)) & 15u) return SKV_ERR_INVALID_ARG;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != ctx->cfg.device && cudaSetDevice(ctx->cfg.device) != cudaSuccess) return SKV_ERR_CUDA;
    skv::Dev d = ctx->d;
    d.layer_sel = layer;
    const cudaError_t e = skv::launch_attend(d, req_ids_dev, B, q_dev, slots_dev, out_dev, lse_dev, sm_scale, stream);
    if (prev >= 0 && prev != ctx->cfg.device) cudaSetDevice(prev);
    if (e != cudaSuccess) {
        skv::set_last_error_message((std::string("skv_attend: ") + cudaGetErrorString(e)).c_str());
        return SKV_ERR_CUDA;
    }
    return SKV_OK;
}

extern "C" skv_status skv_selftest_mma(const void* a_dev, const void* b_dev, float* d_dev, int32_t n, int32_t k,
                                       int32_t b_mn_major, skv_stream_t stream)
{
    if (!a_dev || !b_dev || !d_dev || n < 16 || n > 256 || n % 16 || k < 16 || k > 128 || k % 16)
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
                                                                        n, k, b_mn_major, status);
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
