// Tensor-core kernels of the consumer side: a self-test of the tcgen05 MMA
// path (one 128 x N x K bf16 tile).  The sparse attention over assembled
// slots builds on the same primitives.

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

}  // namespace
}  // namespace skv

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
