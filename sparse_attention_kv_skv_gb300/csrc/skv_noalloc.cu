// skv_assemble_noalloc: the assemble step with its gather work list in a
// static device array instead of context memory, for callers that must not
// allocate device memory at call time.
//
// Who needs it.  Serving engines commonly reserve (nearly) all free HBM for
// their own KV pools and graph memory pools at start-up and then forbid or
// cannot satisfy further cudaMalloc calls; code that runs inside another
// component's stream capture may not allocate either.  Such a caller gets
// the work list from a static array that skv_create has already brought into
// existence on the context's device: CUDA loads a translation unit's device
// code and data lazily, and this file has no kernel that would load it, so
// skv_create looks the array up (noalloc_prepare), which loads it there and
// then.  The pages describe no such entry point; it is a deployment aid.
//
// The array is shared by every call on the device, from every context, and
// keeps the last call's contents.  It needs no clearing: the step's own
// validate kernel resets the work-list counter (context memory) before the
// plan kernel appends to the list, and the gather reads only the entries the
// plan wrote.  Calls that overlap on the GPU -- on different streams, or from
// different contexts -- race on the array.

#include <mutex>
#include <string>
#include <vector>

#include "skv_ctx.cuh"

// Gather work list: one (pool row, hot row) pair per missed token, at most one
// per Top-k entry of the call, so B * L * k must not exceed this.  8 MiB on
// every device that loads the library, held until the process exits.
static constexpr uint32_t kNoAllocMaxEntries = 1u << 20;
static __device__ __align__(256) uint2 g_noalloc_jobs[kNoAllocMaxEntries];

namespace {

// Device address of g_noalloc_jobs, per device ordinal.  In host code the
// name g_noalloc_jobs is only a host-side stand-in for the symbol, never a
// device address, so it is looked up with cudaGetSymbolAddress once per device
// with that device current.
std::mutex g_mu;
std::vector<uint2*> g_jobs_ptr;

cudaError_t jobs_address(int device, uint2** out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if ((int)g_jobs_ptr.size() <= device) g_jobs_ptr.resize(device + 1, nullptr);
    if (!g_jobs_ptr[device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_jobs);
        if (e != cudaSuccess) return e;
        g_jobs_ptr[device] = static_cast<uint2*>(p);
    }
    *out = g_jobs_ptr[device];
    return cudaSuccess;
}

}  // namespace

// Called by skv_create with the context's device current: loads the array on
// that device (its 8 MiB are allocated by the driver now, at create, not at a
// later skv_assemble_noalloc) and caches its address.
cudaError_t skv::noalloc_prepare(int device)
{
    uint2* p = nullptr;
    return jobs_address(device, &p);
}

namespace {

skv_status fail(const std::string& msg, skv_status s)
{
    skv::set_last_error_message(msg.c_str());
    return s;
}

}  // namespace

extern "C" skv_status skv_assemble_noalloc(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B,
                                           const int32_t* topk_dev, int32_t* slots_dev, int32_t* hits_dev,
                                           int32_t* misses_dev, skv_stream_t stream)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch) return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids_dev || !topk_dev || !slots_dev || !hits_dev || !misses_dev) return SKV_ERR_INVALID_ARG;
    const uint64_t entries = (uint64_t)B * ctx->cfg.num_layers * ctx->cfg.topk;
    if (entries > kNoAllocMaxEntries)
        return fail("skv_assemble_noalloc: B*L*k = " + std::to_string(entries) +
                        " exceeds the static work-list capacity of " + std::to_string(kNoAllocMaxEntries) +
                        " entries",
                    SKV_ERR_INVALID_ARG);
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    const int dev = ctx->cfg.device;
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return fail("skv_assemble_noalloc: cudaSetDevice", SKV_ERR_CUDA);
    skv_status st = SKV_OK;
    uint2* jobs = nullptr;
    cudaError_t e = jobs_address(dev, &jobs);
    if (e != cudaSuccess) {
        st = fail(std::string("skv_assemble_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e), SKV_ERR_CUDA);
    } else {
        skv::Dev d = ctx->d;  // the context's state, with the static work list
        d.jobs = jobs;
        if ((e = skv::launch_validate(d, req_ids_dev, B, topk_dev, stream)) != cudaSuccess ||
            (e = skv::launch_plan(d, req_ids_dev, B, topk_dev, slots_dev, hits_dev, misses_dev, false, stream)) !=
                cudaSuccess ||
            (e = skv::launch_gather(d, ctx->gather_grid, stream)) != cudaSuccess)
            st = fail(std::string("skv_assemble_noalloc: kernel launch: ") + cudaGetErrorString(e), SKV_ERR_CUDA);
    }
    if (prev >= 0 && prev != dev) cudaSetDevice(prev);
    return st;
}
