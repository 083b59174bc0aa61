// Lifecycle kernels: request reset (publish / release) and write back.
//
// Pages: KV management follows the request lifecycle publish, acquire, write
// back, release ("XM-Sparse: Netpreme X-Mem ...", section on the SGLang
// HiSparse integration); the complete KV history lives in host memory
// ("Sparse Attention-Driven KVCache Management for Domestic AI Supernodes",
// abstract), so a new token's row is written back to the host pool.

#include "skv_internal.cuh"

namespace skv {
namespace {

// LRU order of a fresh unit: slots 0..S-1 (all last used at clock 0, ties by
// slot index).  Covers units [u0, u0 + nunits).
__global__ void init_lru_kernel(uint16_t* lru, int S, int64_t u0, int64_t nunits, int64_t* len, int32_t* active,
                                int r, int64_t new_len, int new_active)
{
    const int64_t n = nunits * S;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        lru[u0 * S + i] = (uint16_t)(i % S);
    if (r >= 0 && blockIdx.x == 0 && threadIdx.x == 0) {
        len[r] = new_len;
        active[r] = new_active;
    }
}

// write back, phase 1 (one CTA): check every id (in range, active, not
// repeated) and that its pool region has room; on success reserve position
// len[r] for each and advance len.  All or nothing.
__global__ void __launch_bounds__(kLifecycleThreads) write_back_check_kernel(Dev d, const int32_t* __restrict__ req_ids,
                                                                             int n)
{
    __shared__ uint32_t flags;
    if (d.ctl[CTL_ERR] != 0) return;  // sticky error: no-op (phase 2 checks the same word)
    if (threadIdx.x == 0) flags = 0;
    __syncthreads();
    uint32_t f = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int32_t r = req_ids[i];
        if (r < 0 || r >= d.R || d.active[r] == 0) {
            f |= DEVERR_BAD_REQUEST;
            continue;
        }
        for (int j = 0; j < i; ++j)
            if (req_ids[j] == r) f |= DEVERR_BAD_REQUEST;
        if (d.len[r] >= d.T_max) f |= DEVERR_CONTEXT_FULL;
    }
    if (f) atomicOr(&flags, f);
    __syncthreads();
    if (flags) {
        if (threadIdx.x == 0) d.ctl[CTL_ERR] |= flags;
        return;
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int32_t r = req_ids[i];
        const int64_t p = d.len[r];
        d.wb_pos[i] = p;
        d.len[r] = p + 1;
    }
}

// write back, phase 2: row (i, l) -> pool[(r*L + l)*T_max + wb_pos[i]], 16-byte
// chunks, stored through the mapped pool over the host link.
__global__ void __launch_bounds__(kLifecycleThreads) write_back_copy_kernel(Dev d, const int32_t* __restrict__ req_ids,
                                                                            int n, const int4* __restrict__ rows)
{
    if (d.ctl[CTL_ERR] != 0) return;
    const int cpr = d.row_bytes / 16;
    const int64_t total = (int64_t)n * d.L * cpr;
    int4* pool = reinterpret_cast<int4*>(d.pool);
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rowi = c / cpr;  // = i*L + l
        const int w = (int)(c - rowi * cpr);
        const int i = (int)(rowi / d.L), l = (int)(rowi % d.L);
        const int64_t dst_row = ((int64_t)req_ids[i] * d.L + l) * d.T_max + d.wb_pos[i];
        pool[dst_row * cpr + w] = rows[c];
    }
}

// extend, phase 1 (one thread): the request must be active and its pool region
// must have room for n more rows; on success reserve [len, len + n).
__global__ void extend_check_kernel(Dev d, int r, int64_t n)
{
    if (threadIdx.x != 0 || d.ctl[CTL_ERR] != 0) return;  // sticky error: no-op
    uint32_t f = 0;
    if (d.active[r] == 0) f |= DEVERR_BAD_REQUEST;
    else if (d.len[r] + n > d.T_max) f |= DEVERR_CONTEXT_FULL;
    if (f) {
        d.ctl[CTL_ERR] |= f;
        return;
    }
    d.wb_pos[0] = d.len[r];
    d.len[r] += n;
}

// extend, phase 2: rows [L][n][row_bytes] -> pool rows [len, len + n) of each
// layer of request r, 16-byte chunks through the mapped pool.
__global__ void __launch_bounds__(kLifecycleThreads) extend_copy_kernel(Dev d, int r, int64_t n,
                                                                        const int4* __restrict__ rows)
{
    if (d.ctl[CTL_ERR] != 0) return;
    const int cpr = d.row_bytes / 16;
    const int64_t total = (int64_t)d.L * n * cpr;
    const int64_t pos = d.wb_pos[0];
    int4* pool = reinterpret_cast<int4*>(d.pool);
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rowi = c / cpr;  // = l*n + j
        const int w = (int)(c - rowi * cpr);
        const int l = (int)(rowi / n);
        const int64_t j = rowi - (int64_t)l * n;
        pool[(((int64_t)r * d.L + l) * d.T_max + pos + j) * cpr + w] = rows[c];
    }
}

// Candidates of a recency prefetch: for batch entry b (one CTA) and every
// layer of the call, the n newest tokens of request req_ids[b],
// [max(0, len - n), len) ascending, then -1 up to k.  The length is read
// here, on the device, so the window follows write backs and extends earlier
// on the stream.  An id that is not a request gets an all -1 row (the
// validation that follows rejects the call for it).
__global__ void __launch_bounds__(kLifecycleThreads) recent_candidates_kernel(Dev d, const int32_t* __restrict__ req_ids,
                                                                              int n, int32_t* __restrict__ cand)
{
    const int b = blockIdx.x;
    const int32_t r = req_ids[b];
    const int64_t len = r >= 0 && r < d.R ? d.len[r] : 0;
    const int64_t first = len > n ? len - n : 0;
    const int rows = d.layer_sel >= 0 ? 1 : d.L;
    int32_t* out = cand + (size_t)b * rows * d.k;
    for (int i = threadIdx.x; i < rows * d.k; i += blockDim.x) {
        const int64_t t = first + i % d.k;
        out[i] = t < len ? (int32_t)t : -1;
    }
}

}  // namespace

cudaError_t launch_recent_candidates(const Dev& d, const int32_t* req_ids, int B, int n, int32_t* cand, cudaStream_t st)
{
    recent_candidates_kernel<<<B, kLifecycleThreads, 0, st>>>(d, req_ids, n, cand);
    return cudaGetLastError();
}

cudaError_t launch_extend(const Dev& d, int r, int64_t n, const void* rows, cudaStream_t st)
{
    extend_check_kernel<<<1, 32, 0, st>>>(d, r, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t total = (int64_t)d.L * n * (d.row_bytes / 16);
    int64_t g = (total + kLifecycleThreads - 1) / kLifecycleThreads;
    const int grid = (int)(g < 4096 ? g : 4096);
    extend_copy_kernel<<<grid, kLifecycleThreads, 0, st>>>(d, r, n, reinterpret_cast<const int4*>(rows));
    return cudaGetLastError();
}

cudaError_t launch_reset_request(const Dev& d, int r, int64_t len, int active, cudaStream_t st)
{
    const int64_t u0 = (int64_t)r * d.L;
    cudaError_t e;
    if ((e = cudaMemsetAsync(d.tok2slot + u0 * d.T_max, 0xFF, (size_t)d.L * d.T_max * 4, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(d.slot2tok + u0 * d.S, 0xFF, (size_t)d.L * d.S * 4, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(d.ts + u0 * d.S, 0, (size_t)d.L * d.S * 4, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(d.hot + (size_t)u0 * d.S * d.row_bytes, 0, (size_t)d.L * d.S * d.row_bytes, st)) !=
        cudaSuccess)
        return e;
    const int64_t n = (int64_t)d.L * d.S;
    const int grid = (int)((n + kLifecycleThreads - 1) / kLifecycleThreads);
    init_lru_kernel<<<grid, kLifecycleThreads, 0, st>>>(d.lru, d.S, u0, d.L, d.len, d.active, r, len, active);
    return cudaGetLastError();
}

cudaError_t launch_init_lru_all(const Dev& d, cudaStream_t st)
{
    const int64_t n = (int64_t)d.R * d.L * d.S;
    int64_t g = (n + kLifecycleThreads - 1) / kLifecycleThreads;
    const int grid = (int)(g < 65536 ? g : 65536);
    init_lru_kernel<<<grid, kLifecycleThreads, 0, st>>>(d.lru, d.S, 0, (int64_t)d.R * d.L, d.len, d.active, -1, 0, 0);
    return cudaGetLastError();
}

cudaError_t launch_write_back(const Dev& d, const int32_t* req_ids, int n, const void* rows, cudaStream_t st)
{
    write_back_check_kernel<<<1, kLifecycleThreads, 0, st>>>(d, req_ids, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t total = (int64_t)n * d.L * (d.row_bytes / 16);
    int64_t g = (total + kLifecycleThreads - 1) / kLifecycleThreads;
    const int grid = (int)(g < 4096 ? g : 4096);
    write_back_copy_kernel<<<grid, kLifecycleThreads, 0, st>>>(d, req_ids, n, reinterpret_cast<const int4*>(rows));
    return cudaGetLastError();
}

}  // namespace skv
