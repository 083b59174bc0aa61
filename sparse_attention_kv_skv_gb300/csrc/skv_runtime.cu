// Host runtime behind the C ABI (include/skv.h): context creation and memory
// layout, the request table, argument checks, and the stream-ordered launch
// sequences of each call.  No call after skv_create allocates memory.
//
// Pages: the SparseKVCacheManager consists of host storage, a device cache and
// an index mapping ("Sparse Attention-Driven KVCache Management for Domestic
// AI Supernodes", agenda item 2); requests go through publish, acquire, write
// back and release ("XM-Sparse: Netpreme X-Mem ...", section on the SGLang
// HiSparse integration).

#include <dirent.h>
#include <sys/syscall.h>
#include <unistd.h>

#include <algorithm>
#include <cctype>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "skv_ctx.cuh"

using skv::Dev;

namespace {

thread_local std::string g_last_cuda_error;

skv_status cuda_fail(cudaError_t e, const char* what)
{
    g_last_cuda_error = std::string(what) + ": " + cudaGetErrorString(e);
    return SKV_ERR_CUDA;
}

#define SKV_CUDA(call)                                       \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);  \
    } while (0)

// Makes the context's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool is_device_pointer(const void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

void free_pool(skv_ctx* x);

// The device address of host memory the device can write directly (pinned
// and mapped into its address space, e.g. cudaHostAlloc memory); nullptr for
// anything else (pageable host memory, device memory).
void* device_view_of_host(void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

void free_ctx(skv_ctx* c)
{
    if (!c) return;
    cudaFree(c->d.tok2slot);
    cudaFree(c->d.slot2tok);
    cudaFree(c->d.ts);
    cudaFree(c->d.lru);
    cudaFree(c->d.hot);
    cudaFree(c->d.len);
    cudaFree(c->d.active);
    cudaFree(c->d.ctl);
    cudaFree(c->d.stats);
    cudaFree(c->d.wb_pos);
    cudaFree(c->st_req);
    cudaFree(c->st_topk);
    cudaFree(c->st_slots);
    cudaFree(c->st_hits);
    cudaFree(c->st_misses);
    if (c->host_word) cudaFreeHost(c->host_word);
    free_pool(c);
    delete c;
}

// ---------------------------------------------------------------------------
// NUMA placement of the host pool.  On a host with several memory nodes (two
// Grace CPUs to a tray, each linked to its own GPUs), a pool on the far node
// makes every gather cross the CPU-to-CPU link as well.  The node nearest the
// GPU is the one whose CPUs are the PCI device's local CPUs (sysfs, read
// only); the pool is allocated under a preferred-node memory policy for that
// node, and the caller's policy is restored afterwards.
// ---------------------------------------------------------------------------
constexpr int kMaxNodes = 1024;  // node ids this code handles (bits of the masks below)
constexpr long kMpolDefault = 0, kMpolPreferred = 1;

std::string read_text(const std::string& path)
{
    std::string out;
    FILE* f = std::fopen(path.c_str(), "r");
    if (!f) return out;
    char buf[4096];
    size_t n;
    while ((n = std::fread(buf, 1, sizeof buf, f)) > 0) out.append(buf, n);
    std::fclose(f);
    while (!out.empty() && std::isspace((unsigned char)out.back())) out.pop_back();
    return out;
}

// "0-3,8,10-11" -> {0,1,2,3,8,10,11}; false on a malformed list
bool parse_cpulist(const std::string& s, std::vector<int>& cpus)
{
    cpus.clear();
    size_t i = 0;
    while (i < s.size()) {
        char* end = nullptr;
        const long a = std::strtol(s.c_str() + i, &end, 10);
        if (end == s.c_str() + i || a < 0) return false;
        i = (size_t)(end - s.c_str());
        long b = a;
        if (i < s.size() && s[i] == '-') {
            ++i;
            b = std::strtol(s.c_str() + i, &end, 10);
            if (end == s.c_str() + i || b < a || b - a > 65536) return false;
            i = (size_t)(end - s.c_str());
        }
        for (long c = a; c <= b; ++c) cpus.push_back((int)c);
        if (i < s.size()) {
            if (s[i] != ',') return false;
            ++i;
        }
    }
    return true;
}

// sysfs name of a PCI bus id as CUDA prints it ("0000:01:00.0", or with an
// 8-digit domain): lower case, 4-digit domain
std::string sysfs_bus_id(const char* id)
{
    std::string s(id);
    for (auto& c : s) c = (char)std::tolower((unsigned char)c);
    const size_t colon = s.find(':');
    if (colon != std::string::npos && colon > 4) s = s.substr(colon - 4);
    return s;
}

int host_node_for_pci(const std::string& sysfs, const std::string& bus_id)
{
    const std::string dev = sysfs + "/bus/pci/devices/" + bus_id;
    std::vector<int> local;
    const bool have_local = parse_cpulist(read_text(dev + "/local_cpulist"), local) && !local.empty();
    const std::string nodes_dir = sysfs + "/devices/system/node";
    int best = -1;
    size_t best_overlap = 0;
    std::vector<int> with_cpus;
    if (DIR* dir = opendir(nodes_dir.c_str())) {
        while (dirent* e = readdir(dir)) {
            if (std::strncmp(e->d_name, "node", 4) != 0 || !std::isdigit((unsigned char)e->d_name[4])) continue;
            const int node = std::atoi(e->d_name + 4);
            std::vector<int> cpus;
            if (!parse_cpulist(read_text(nodes_dir + "/" + e->d_name + "/cpulist"), cpus) || cpus.empty()) continue;
            with_cpus.push_back(node);
            if (!have_local) continue;
            size_t overlap = 0;
            for (int c : cpus) overlap += std::count(local.begin(), local.end(), c) > 0;
            if (overlap > best_overlap || (overlap == best_overlap && overlap > 0 && node < best)) {
                best_overlap = overlap;
                best = node;
            }
        }
        closedir(dir);
    }
    if (best >= 0) return best;
    // no local CPU list: the device's own node, if that node has CPUs (a node
    // without CPUs may be GPU memory itself)
    const std::string nn = read_text(dev + "/numa_node");
    if (!nn.empty()) {
        const int node = std::atoi(nn.c_str());
        if (node >= 0 && std::find(with_cpus.begin(), with_cpus.end(), node) != with_cpus.end()) return node;
    }
    return -1;
}

// The calling thread's memory policy set to "prefer `node`" for the lifetime
// of the object, then put back as it was.  Does nothing for node < 0.
struct PreferNode {
    long old_mode = kMpolDefault;
    unsigned long old_mask[kMaxNodes / 64] = {};
    bool active = false;
    explicit PreferNode(int node)
    {
        if (node < 0 || node >= kMaxNodes) return;
        int mode = 0;
        if (syscall(SYS_get_mempolicy, &mode, old_mask, (unsigned long)kMaxNodes + 1, nullptr, 0ul) != 0) return;
        old_mode = mode;
        unsigned long mask[kMaxNodes / 64] = {};
        mask[node / 64] = 1ul << (node % 64);
        active = syscall(SYS_set_mempolicy, kMpolPreferred, mask, (unsigned long)kMaxNodes + 1) == 0;
    }
    ~PreferNode()
    {
        if (active) syscall(SYS_set_mempolicy, old_mode, old_mask, (unsigned long)kMaxNodes + 1);
    }
};

// The node holding most of a sample of pages of [base, base + bytes), and the
// share of the sample there; -1 if the kernel reports no node for them.
void sample_placement(const void* base, size_t bytes, int* node, float* frac)
{
    *node = -1;
    *frac = 0.0f;
    const long page = sysconf(_SC_PAGESIZE);
    if (!base || bytes == 0 || page <= 0) return;
    constexpr int kSamples = 64;
    void* pages[kSamples];
    int status[kSamples];
    int n = 0;
    for (int i = 0; i < kSamples; ++i) {
        const size_t off = (size_t)((double)bytes * i / kSamples) / (size_t)page * (size_t)page;
        if (off < bytes) pages[n++] = (void*)((const char*)base + off);
    }
    if (syscall(SYS_move_pages, 0, (unsigned long)n, pages, nullptr, status, 0) != 0) return;
    std::vector<int> count;
    for (int i = 0; i < n; ++i)
        if (status[i] >= 0 && status[i] < kMaxNodes) {
            if ((int)count.size() <= status[i]) count.resize(status[i] + 1, 0);
            ++count[status[i]];
        }
    if (count.empty()) return;
    const int best = (int)(std::max_element(count.begin(), count.end()) - count.begin());
    *node = best;
    *frac = (float)count[best] / (float)n;
}

// The node the pool of a context on `device` should live on: SKV_POOL_NODE if
// set (-1: no preference), else the host node nearest the device.
int pool_node_for_device(int device)
{
    if (const char* v = std::getenv("SKV_POOL_NODE")) return std::atoi(v);
    char bus[64] = {};
    if (cudaDeviceGetPCIBusId(bus, (int)sizeof bus, device) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return host_node_for_pci("/sys", sysfs_bus_id(bus));
}

// The host pool: pinned and mapped for the device with cudaHostAlloc.  (A
// huge-page mapping registered with cudaHostRegister was tried: a stand-alone
// gather over it starts faster, but once the CPU writes the published rows into
// the registered range, device reads of it run one to two orders of magnitude
// below link speed for many steps on GB300, so it is not used.)
cudaError_t alloc_pool(skv_ctx* x, size_t bytes)
{
    try {  // no C++ exception may leave a C entry point: without a topology, no preference
        x->pool_node_wanted = pool_node_for_device(x->cfg.device);
    } catch (...) {
        x->pool_node_wanted = -1;
    }
    cudaError_t e;
    {
        PreferNode scope(x->pool_node_wanted);
        e = cudaHostAlloc((void**)&x->pool_host, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    }
    if (e == cudaSuccess) {
        try {
            sample_placement(x->pool_host, bytes, &x->pool_node_seen, &x->pool_node_frac);
        } catch (...) {
            x->pool_node_seen = -1;
        }
    }
    return e;
}

void free_pool(skv_ctx* x)
{
    if (x->pool_host) cudaFreeHost(x->pool_host);
    x->pool_host = nullptr;
}

// Parallel host memcpy for large publishes from host memory.
void host_copy(uint8_t* dst, const uint8_t* src, size_t n)
{
    const size_t chunk = (size_t)64 << 20;
    if (n <= chunk) {
        std::memcpy(dst, src, n);
        return;
    }
    unsigned nt = std::thread::hardware_concurrency();
    nt = nt < 1 ? 1 : (nt > 16 ? 16 : nt);
    std::vector<std::thread> th;
    const size_t per = (n + nt - 1) / nt;
    for (unsigned i = 0; i < nt; ++i) {
        const size_t o = (size_t)i * per;
        if (o >= n) break;
        const size_t len = n - o < per ? n - o : per;
        try {  // no C++ exception may leave a C entry point
            th.emplace_back([=] { std::memcpy(dst + o, src + o, len); });
        } catch (...) {  // no thread to spare: copy this share here
            std::memcpy(dst + o, src + o, len);
        }
    }
    for (auto& t : th) t.join();
}

// A timing event: during stream capture it must become an external event
// record node of the graph (a plain record would only be a dependency marker);
// outside capture it is an ordinary record.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return e;
    if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    return cudaEventRecord(ev, stream);
}

// Test hook for the allocation-failure path of skv_create: when the
// environment variable SKV_TEST_FAIL_ALLOC=n (n >= 1) is set, the n-th
// allocation of a create call fails with cudaErrorMemoryAllocation without
// being attempted.  Read at every create; unset (or 0) it does nothing.  Only
// tests set it: a real out-of-memory on a shared GPU is not something to
// provoke.
struct AllocFault {
    long fail_at = 0, seen = 0;
    AllocFault()
    {
        const char* v = std::getenv("SKV_TEST_FAIL_ALLOC");
        if (v) fail_at = std::strtol(v, nullptr, 10);
    }
    bool next() { return fail_at > 0 && ++seen == fail_at; }
};

}  // namespace

void skv::set_last_error_message(const char* msg) { g_last_cuda_error = msg; }

extern "C" {

const char* skv_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

const char* skv_status_string(skv_status s)
{
    switch (s) {
        case SKV_OK: return "SKV_OK";
        case SKV_ERR_INVALID_ARG: return "SKV_ERR_INVALID_ARG";
        case SKV_ERR_OOM: return "SKV_ERR_OOM";
        case SKV_ERR_BAD_REQUEST: return "SKV_ERR_BAD_REQUEST";
        case SKV_ERR_NO_FREE_REQUEST: return "SKV_ERR_NO_FREE_REQUEST";
        case SKV_ERR_CONTEXT_FULL: return "SKV_ERR_CONTEXT_FULL";
        case SKV_ERR_CUDA: return "SKV_ERR_CUDA";
    }
    return "unknown skv_status";
}

skv_status skv_create(const skv_config* cfg, skv_ctx** out)
{
    if (!cfg || !out) return SKV_ERR_INVALID_ARG;
    *out = nullptr;
    const skv_config c = *cfg;
    if (c.max_requests < 1 || c.num_layers < 1 || c.max_context < 1 || c.row_bytes < 16 || c.row_bytes % 16 != 0 ||
        c.row_bytes > 65536 ||
        c.topk < 1 || c.topk > skv::kMaxTopk || c.hot_slots < c.topk || c.hot_slots > skv::kMaxSlots ||
        c.max_batch < 1 || c.device < 0)
        return SKV_ERR_INVALID_ARG;
    const uint64_t units = (uint64_t)c.max_requests * (uint64_t)c.num_layers;
    if (units * (uint64_t)c.max_context >= (1ull << 32) || units * (uint64_t)c.hot_slots >= (1ull << 32))
        return SKV_ERR_INVALID_ARG;
    if ((uint64_t)c.max_batch * c.num_layers * c.topk >= (1ull << 31) || (uint64_t)c.max_batch * c.num_layers >= (1ull << 31))
        return SKV_ERR_INVALID_ARG;

    DeviceGuard g(c.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    skv_ctx* x = new (std::nothrow) skv_ctx();
    if (!x) return SKV_ERR_OOM;
    x->cfg = c;
    try {  // no C++ exception may leave a C entry point
        x->active_h.assign(c.max_requests, 0);
    } catch (const std::bad_alloc&) {
        delete x;
        return SKV_ERR_OOM;
    }
    Dev& d = x->d;
    d.R = c.max_requests;
    d.L = c.num_layers;
    d.k = c.topk;
    d.S = c.hot_slots;
    d.row_bytes = c.row_bytes;
    d.T_max = c.max_context;
    d.layer_sel = -1;

    auto fail = [&](cudaError_t e, const char* what) {
        skv_status s = (e == cudaErrorMemoryAllocation) ? SKV_ERR_OOM : cuda_fail(e, what);
        if (e == cudaErrorMemoryAllocation) g_last_cuda_error = std::string(what) + ": out of memory";
        cudaGetLastError();
        free_ctx(x);
        return s;
    };
#define SKV_TRY(call)                                \
    do {                                             \
        cudaError_t e_ = (call);                     \
        if (e_ != cudaSuccess) return fail(e_, #call); \
    } while (0)
    // an allocation, unless the test hook makes it fail
    AllocFault fault;
#define SKV_ALLOC(call) SKV_TRY(fault.next() ? cudaErrorMemoryAllocation : (call))

    const size_t pool_bytes = (size_t)units * c.max_context * c.row_bytes;
    SKV_ALLOC(alloc_pool(x, pool_bytes));
    SKV_TRY(cudaHostGetDevicePointer((void**)&d.pool, x->pool_host, 0));
    SKV_ALLOC(cudaHostAlloc((void**)&x->host_word, 64, cudaHostAllocDefault));
    SKV_ALLOC(cudaMalloc(&d.tok2slot, (size_t)units * c.max_context * 4));
    SKV_ALLOC(cudaMalloc(&d.slot2tok, (size_t)units * c.hot_slots * 4));
    SKV_ALLOC(cudaMalloc(&d.ts, (size_t)units * c.hot_slots * 4));
    SKV_ALLOC(cudaMalloc(&d.lru, (size_t)units * c.hot_slots * 2));
    SKV_ALLOC(cudaMalloc(&d.hot, (size_t)units * c.hot_slots * c.row_bytes));
    SKV_ALLOC(cudaMalloc(&d.len, (size_t)c.max_requests * 8));
    SKV_ALLOC(cudaMalloc(&d.active, (size_t)c.max_requests * 4));
    SKV_ALLOC(cudaMalloc(&d.ctl, skv::CTL_WORDS * 4));
    SKV_ALLOC(cudaMalloc(&d.stats, skv::STAT_WORDS * 8));
    const size_t step_entries = (size_t)c.max_batch * c.num_layers * c.topk;
    d.jobs = nullptr;  // only skv_assemble_noalloc queues gather jobs, into its static array
    SKV_ALLOC(cudaMalloc(&d.wb_pos, (size_t)c.max_batch * 8));
    SKV_ALLOC(cudaMalloc(&x->st_req, (size_t)c.max_batch * 4));
    SKV_ALLOC(cudaMalloc(&x->st_topk, step_entries * 4));
    SKV_ALLOC(cudaMalloc(&x->st_slots, step_entries * 4));
    SKV_ALLOC(cudaMalloc(&x->st_hits, (size_t)c.max_batch * c.num_layers * 4));
    SKV_ALLOC(cudaMalloc(&x->st_misses, (size_t)c.max_batch * c.num_layers * 4));

    SKV_TRY(cudaMemset(d.tok2slot, 0xFF, (size_t)units * c.max_context * 4));
    SKV_TRY(cudaMemset(d.slot2tok, 0xFF, (size_t)units * c.hot_slots * 4));
    SKV_TRY(cudaMemset(d.ts, 0, (size_t)units * c.hot_slots * 4));
    SKV_TRY(cudaMemset(d.hot, 0, (size_t)units * c.hot_slots * c.row_bytes));
    SKV_TRY(cudaMemset(d.len, 0, (size_t)c.max_requests * 8));
    SKV_TRY(cudaMemset(d.active, 0, (size_t)c.max_requests * 4));
    SKV_TRY(cudaMemset(d.ctl, 0, skv::CTL_WORDS * 4));
    SKV_TRY(cudaMemset(d.stats, 0, skv::STAT_WORDS * 8));
    SKV_TRY(skv::launch_init_lru_all(d, 0));
    SKV_TRY(skv::prepare_step_kernels(c.topk, c.hot_slots, &x->gather_grid));
    SKV_TRY(skv::prepare_attend(&x->device_sms));
    SKV_TRY(skv::noalloc_prepare(c.device));
    SKV_TRY(cudaDeviceSynchronize());
#undef SKV_ALLOC
#undef SKV_TRY
    *out = x;
    return SKV_OK;
}

skv_status skv_destroy(skv_ctx* ctx)
{
    if (!ctx) return SKV_OK;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaDeviceSynchronize();
    free_ctx(ctx);
    return SKV_OK;
}

skv_status skv_publish(skv_ctx* ctx, const void* rows, int64_t T, int32_t* out_req, skv_stream_t stream)
{
    if (!ctx || !out_req || T < 0) return SKV_ERR_INVALID_ARG;
    if (T > ctx->cfg.max_context) return SKV_ERR_CONTEXT_FULL;
    int32_t r = -1;
    for (int32_t i = 0; i < ctx->cfg.max_requests; ++i)
        if (!ctx->active_h[i]) {
            r = i;
            break;
        }
    if (r < 0) return SKV_ERR_NO_FREE_REQUEST;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    const Dev& d = ctx->d;
    const size_t rb = (size_t)d.row_bytes;
    if (rows && T > 0) {
        if (is_device_pointer(rows)) {
            for (int l = 0; l < d.L; ++l)
                SKV_CUDA(cudaMemcpyAsync(ctx->pool_host + (((size_t)r * d.L + l) * d.T_max) * rb,
                                         static_cast<const uint8_t*>(rows) + (size_t)l * T * rb, (size_t)T * rb,
                                         cudaMemcpyDefault, stream));
        } else {
            SKV_CUDA(cudaStreamSynchronize(stream));
            for (int l = 0; l < d.L; ++l)
                host_copy(ctx->pool_host + (((size_t)r * d.L + l) * d.T_max) * rb,
                          static_cast<const uint8_t*>(rows) + (size_t)l * T * rb, (size_t)T * rb);
        }
    }
    SKV_CUDA(skv::launch_reset_request(d, r, T, 1, stream));
    ctx->active_h[r] = 1;
    *out_req = r;
    return SKV_OK;
}

skv_status skv_release(skv_ctx* ctx, int32_t req, skv_stream_t stream)
{
    if (!ctx) return SKV_ERR_INVALID_ARG;
    if (req < 0 || req >= ctx->cfg.max_requests || !ctx->active_h[req]) return SKV_ERR_BAD_REQUEST;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    SKV_CUDA(skv::launch_reset_request(ctx->d, req, 0, 0, stream));
    ctx->active_h[req] = 0;
    return SKV_OK;
}

skv_status skv_write_back(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t n, const void* rows_dev,
                          skv_stream_t stream)
{
    if (!ctx || n < 0 || n > ctx->cfg.max_batch) return SKV_ERR_INVALID_ARG;
    if (n == 0) return SKV_OK;
    if (!req_ids_dev || !rows_dev || (reinterpret_cast<uintptr_t>(rows_dev) & 15u)) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    SKV_CUDA(skv::launch_write_back(ctx->d, req_ids_dev, n, rows_dev, stream));
    return SKV_OK;
}

}  // extern "C"

namespace {
// The launch sequence of one assemble call over the units described by `d`
// (all layers, or the one in d.layer_sel).  `timed`: record the caller's
// events around the call's two kernels (assemble calls only, not prefetches).
// The first event goes before validation, not between the two kernels: a
// record there would keep the fused kernel from starting while validation
// runs (a programmatic dependent launch must follow its primary directly).
skv_status assemble_impl(skv_ctx* ctx, const Dev& d, const int32_t* req_ids_dev, int32_t B, const int32_t* topk_dev,
                         int32_t* slots_dev, int32_t* hits_dev, int32_t* misses_dev, cudaStream_t stream,
                         bool timed = true)
{
    if (timed && ctx->ev_before) SKV_CUDA(record_event(ctx->ev_before, stream));
    SKV_CUDA(skv::launch_validate(d, req_ids_dev, B, topk_dev, stream));
    SKV_CUDA(skv::launch_plan_gather(d, req_ids_dev, B, topk_dev, slots_dev, hits_dev, misses_dev, ctx->device_sms,
                                     stream));
    if (timed && ctx->ev_after) SKV_CUDA(record_event(ctx->ev_after, stream));
    return SKV_OK;
}
}  // namespace

extern "C" {

skv_status skv_extend(skv_ctx* ctx, int32_t req, const void* rows, int64_t n, skv_stream_t stream)
{
    if (!ctx || n < 0) return SKV_ERR_INVALID_ARG;
    if (req < 0 || req >= ctx->cfg.max_requests || !ctx->active_h[req]) return SKV_ERR_BAD_REQUEST;
    if (n == 0) return SKV_OK;
    if (!rows || (reinterpret_cast<uintptr_t>(rows) & 15u)) return SKV_ERR_INVALID_ARG;
    if (n > ctx->cfg.max_context) return SKV_ERR_CONTEXT_FULL;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    SKV_CUDA(skv::launch_extend(ctx->d, req, n, rows, stream));
    return SKV_OK;
}

skv_status skv_assemble(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B, const int32_t* topk_dev,
                        int32_t* slots_dev, int32_t* hits_dev, int32_t* misses_dev, skv_stream_t stream)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch) return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids_dev || !topk_dev || !slots_dev || !hits_dev || !misses_dev) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    return assemble_impl(ctx, ctx->d, req_ids_dev, B, topk_dev, slots_dev, hits_dev, misses_dev, stream);
}

skv_status skv_assemble_layer(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B, int32_t layer,
                              const int32_t* topk_dev, int32_t* slots_dev, int32_t* hits_dev, int32_t* misses_dev,
                              skv_stream_t stream)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch || layer < 0 || layer >= ctx->cfg.num_layers)
        return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids_dev || !topk_dev || !slots_dev || !hits_dev || !misses_dev) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    Dev d = ctx->d;
    d.layer_sel = layer;
    return assemble_impl(ctx, d, req_ids_dev, B, topk_dev, slots_dev, hits_dev, misses_dev, stream);
}

skv_status skv_prefetch(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B, int32_t layer, const int32_t* cand_dev,
                        int32_t* hits_dev, int32_t* misses_dev, skv_stream_t stream)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch || layer < -1 || layer >= ctx->cfg.num_layers)
        return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids_dev || !cand_dev) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    Dev d = ctx->d;
    d.layer_sel = layer;
    return assemble_impl(ctx, d, req_ids_dev, B, cand_dev, ctx->st_slots, hits_dev ? hits_dev : ctx->st_hits,
                         misses_dev ? misses_dev : ctx->st_misses, stream, false);
}

skv_status skv_prefetch_recent(skv_ctx* ctx, const int32_t* req_ids_dev, int32_t B, int32_t layer, int32_t n,
                               int32_t* hits_dev, int32_t* misses_dev, skv_stream_t stream)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch || layer < -1 || layer >= ctx->cfg.num_layers || n < 0 ||
        n > ctx->cfg.topk)
        return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids_dev) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    Dev d = ctx->d;
    d.layer_sel = layer;
    SKV_CUDA(skv::launch_recent_candidates(d, req_ids_dev, B, n, ctx->st_topk, stream));
    return assemble_impl(ctx, d, req_ids_dev, B, ctx->st_topk, ctx->st_slots, hits_dev ? hits_dev : ctx->st_hits,
                         misses_dev ? misses_dev : ctx->st_misses, stream, false);
}

skv_status skv_assemble_host(skv_ctx* ctx, const int32_t* req_ids, int32_t B, const int32_t* topk, int32_t* slots,
                             int32_t* hits, int32_t* misses, skv_stream_t stream)
{
    if (!ctx || B < 0 || B > ctx->cfg.max_batch) return SKV_ERR_INVALID_ARG;
    if (B == 0) return SKV_OK;
    if (!req_ids || !topk || !slots || !hits || !misses) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    const size_t units = (size_t)B * ctx->cfg.num_layers;
    const size_t entries = units * ctx->cfg.topk;
    SKV_CUDA(cudaMemcpyAsync(ctx->st_req, req_ids, (size_t)B * 4, cudaMemcpyHostToDevice, stream));
    SKV_CUDA(cudaMemcpyAsync(ctx->st_topk, topk, entries * 4, cudaMemcpyHostToDevice, stream));
    // Outputs in pinned host memory the device can address are written by the kernels themselves,
    // through the host link in the direction the gather does not use; the others go through the
    // context's staging buffers and a copy back.
    int32_t* d_slots = static_cast<int32_t*>(device_view_of_host(slots));
    int32_t* d_hits = static_cast<int32_t*>(device_view_of_host(hits));
    int32_t* d_misses = static_cast<int32_t*>(device_view_of_host(misses));
    skv_status s = skv_assemble(ctx, ctx->st_req, B, ctx->st_topk, d_slots ? d_slots : ctx->st_slots,
                                d_hits ? d_hits : ctx->st_hits, d_misses ? d_misses : ctx->st_misses, stream);
    if (s != SKV_OK) return s;
    if (!d_slots) SKV_CUDA(cudaMemcpyAsync(slots, ctx->st_slots, entries * 4, cudaMemcpyDeviceToHost, stream));
    if (!d_hits) SKV_CUDA(cudaMemcpyAsync(hits, ctx->st_hits, units * 4, cudaMemcpyDeviceToHost, stream));
    if (!d_misses) SKV_CUDA(cudaMemcpyAsync(misses, ctx->st_misses, units * 4, cudaMemcpyDeviceToHost, stream));
    SKV_CUDA(cudaStreamSynchronize(stream));
    return SKV_OK;
}

skv_status skv_get_device_error(skv_ctx* ctx, int32_t* bits, skv_stream_t stream)
{
    if (!ctx || !bits) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    SKV_CUDA(cudaMemcpyAsync(ctx->host_word, ctx->d.ctl + skv::CTL_ERR, 4, cudaMemcpyDeviceToHost, stream));
    SKV_CUDA(cudaMemsetAsync(ctx->d.ctl + skv::CTL_ERR, 0, 4, stream));
    SKV_CUDA(cudaStreamSynchronize(stream));
    *bits = (int32_t)ctx->host_word[0];
    return SKV_OK;
}

skv_status skv_hot_buffer(skv_ctx* ctx, void** base, int64_t* unit_stride_bytes)
{
    if (!ctx) return SKV_ERR_INVALID_ARG;
    if (base) *base = ctx->d.hot;
    if (unit_stride_bytes) *unit_stride_bytes = (int64_t)ctx->d.S * ctx->d.row_bytes;
    return SKV_OK;
}

skv_status skv_pool_rows(skv_ctx* ctx, void** host_base)
{
    if (!ctx || !host_base) return SKV_ERR_INVALID_ARG;
    *host_base = ctx->pool_host;
    return SKV_OK;
}

skv_status skv_export_state(skv_ctx* ctx, int32_t req, int32_t* slot2tok, uint32_t* ts, int32_t* tok2slot,
                            int32_t* lru, int64_t* len, int32_t* active, skv_stream_t stream)
{
    if (!ctx) return SKV_ERR_INVALID_ARG;
    if (req < 0 || req >= ctx->cfg.max_requests) return SKV_ERR_BAD_REQUEST;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    const Dev& d = ctx->d;
    const size_t u0 = (size_t)req * d.L;
    const size_t ns = (size_t)d.L * d.S;
    SKV_CUDA(cudaStreamSynchronize(stream));
    if (slot2tok) SKV_CUDA(cudaMemcpy(slot2tok, d.slot2tok + u0 * d.S, ns * 4, cudaMemcpyDeviceToHost));
    if (ts) SKV_CUDA(cudaMemcpy(ts, d.ts + u0 * d.S, ns * 4, cudaMemcpyDeviceToHost));
    if (tok2slot) SKV_CUDA(cudaMemcpy(tok2slot, d.tok2slot + u0 * d.T_max, (size_t)d.L * d.T_max * 4,
                                      cudaMemcpyDeviceToHost));
    if (lru) {
        std::vector<uint16_t> tmp;
        try {  // no C++ exception may leave a C entry point
            tmp.resize(ns);
        } catch (const std::bad_alloc&) {
            return SKV_ERR_OOM;
        }
        SKV_CUDA(cudaMemcpy(tmp.data(), d.lru + u0 * d.S, ns * 2, cudaMemcpyDeviceToHost));
        for (size_t i = 0; i < ns; ++i) lru[i] = tmp[i];
    }
    if (len) SKV_CUDA(cudaMemcpy(len, d.len + req, 8, cudaMemcpyDeviceToHost));
    if (active) SKV_CUDA(cudaMemcpy(active, d.active + req, 4, cudaMemcpyDeviceToHost));
    return SKV_OK;
}

skv_status skv_export_hot(skv_ctx* ctx, int32_t req, void* host_dst, skv_stream_t stream)
{
    if (!ctx || !host_dst) return SKV_ERR_INVALID_ARG;
    if (req < 0 || req >= ctx->cfg.max_requests) return SKV_ERR_BAD_REQUEST;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    const Dev& d = ctx->d;
    SKV_CUDA(cudaStreamSynchronize(stream));
    SKV_CUDA(cudaMemcpy(host_dst, d.hot + (size_t)req * d.L * d.S * d.row_bytes, (size_t)d.L * d.S * d.row_bytes,
                        cudaMemcpyDeviceToHost));
    return SKV_OK;
}

skv_status skv_get_clock(skv_ctx* ctx, uint32_t* clock, skv_stream_t stream)
{
    if (!ctx || !clock) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    SKV_CUDA(cudaStreamSynchronize(stream));
    SKV_CUDA(cudaMemcpy(clock, ctx->d.ctl + skv::CTL_CLOCK, 4, cudaMemcpyDeviceToHost));
    return SKV_OK;
}

skv_status skv_get_stats(skv_ctx* ctx, uint64_t* calls, uint64_t* hits, uint64_t* misses, skv_stream_t stream)
{
    if (!ctx) return SKV_ERR_INVALID_ARG;
    DeviceGuard g(ctx->cfg.device);
    if (!g.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    unsigned long long st[skv::STAT_WORDS];
    SKV_CUDA(cudaStreamSynchronize(stream));
    SKV_CUDA(cudaMemcpy(st, ctx->d.stats, sizeof(st), cudaMemcpyDeviceToHost));
    if (calls) *calls = st[skv::STAT_CALLS];
    if (hits) *hits = st[skv::STAT_HITS];
    if (misses) *misses = st[skv::STAT_MISSES];
    return SKV_OK;
}

skv_status skv_pool_placement(skv_ctx* ctx, int32_t* wanted_node, int32_t* seen_node, float* seen_frac)
{
    if (!ctx) return SKV_ERR_INVALID_ARG;
    if (wanted_node) *wanted_node = ctx->pool_node_wanted;
    if (seen_node) *seen_node = ctx->pool_node_seen;
    if (seen_frac) *seen_frac = ctx->pool_node_frac;
    return SKV_OK;
}

skv_status skv_host_node_for_pci(const char* sysfs_root, const char* pci_bus_id, int32_t* node)
{
    if (!pci_bus_id || !node) return SKV_ERR_INVALID_ARG;
    try {  // no C++ exception may leave a C entry point
        *node = host_node_for_pci(sysfs_root ? sysfs_root : "/sys", sysfs_bus_id(pci_bus_id));
    } catch (...) {
        return SKV_ERR_OOM;
    }
    return SKV_OK;
}

skv_status skv_set_gather_events(skv_ctx* ctx, skv_event_t before, skv_event_t after)
{
    if (!ctx || (before == nullptr) != (after == nullptr)) return SKV_ERR_INVALID_ARG;
    ctx->ev_before = reinterpret_cast<cudaEvent_t>(before);
    ctx->ev_after = reinterpret_cast<cudaEvent_t>(after);
    return SKV_OK;
}

}  // extern "C"
