// Internal declarations shared by the library's translation units: the
// device-state descriptor and the kernel launchers.  Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace skv {

constexpr int kMaxTopk = 4096;    // k limit (plan kernel keeps <= 8 entries per thread)
constexpr int kMaxSlots = 16384;  // S limit (uint16 LRU entries, shared-memory budget)
constexpr int kPlanThreads = 512;
constexpr int kValidateThreads = 512;
constexpr int kGatherThreads = 256;
constexpr int kLifecycleThreads = 256;

// Control words in device memory.
enum : int {
    CTL_CLOCK = 0,     // step clock: successful assemble calls
    CTL_ERR = 1,       // sticky error bits (SKV_DEVERR_*)
    CTL_ERR_CALL = 2,  // error bits found by the running assemble call, committed by the gather kernel
    CTL_JOBS = 3,      // rows queued for the gather by the running assemble call (job-list path)
    CTL_DONE = 4,      // CTAs of the fused plan+gather kernel that have finished (last one commits)
    CTL_WORDS = 5
};
enum : int { STAT_CALLS = 0, STAT_HITS = 1, STAT_MISSES = 2, STAT_WORDS = 3 };

enum : uint32_t {
    DEVERR_BAD_REQUEST = 1,
    DEVERR_BAD_INDEX = 2,
    DEVERR_DUPLICATE = 4,
    DEVERR_CONTEXT_FULL = 8,
    DEVERR_TIMEOUT = 16  // a tensor-core product did not signal completion within its bounded wait
};

// Everything a kernel needs to find the state of unit u = r*L + l.
struct Dev {
    int32_t R, L, k, S, row_bytes;
    int64_t T_max;
    int32_t* tok2slot;     // [R*L][T_max], -1 = not resident
    int32_t* slot2tok;     // [R*L][S], -1 = empty
    uint32_t* ts;          // [R*L][S], last-use clock
    uint16_t* lru;         // [R*L][S], slots by (ts, slot), least recent first
    uint8_t* hot;          // [R*L][S][row_bytes], device cache
    uint8_t* pool;         // [R*L][T_max][row_bytes], mapped host pool (device address)
    int64_t* len;          // [R]
    int32_t* active;       // [R]
    uint32_t* ctl;         // [CTL_WORDS]
    unsigned long long* stats;  // [STAT_WORDS]
    uint2* jobs;           // gather work list: (source pool row, destination hot row)
    int64_t* wb_pos;       // [max_batch] write-back target positions
    int32_t layer_sel;     // -1: a call covers all L layers (CTA = b*L + l); else only this layer (CTA = b)
};

// CTAs (units) of one assemble call.
inline int call_units(const Dev& d, int B) { return d.layer_sel >= 0 ? B : B * d.L; }

// Shared-memory bytes the plan kernel needs for (k, S).
size_t plan_smem_bytes(int k, int S);
size_t validate_smem_bytes(int k);

// Step kernels (assemble).
cudaError_t launch_validate(const Dev& d, const int32_t* req_ids, int B, const int32_t* topk, cudaStream_t st);
// plan with a global work list (copied by launch_gather); pdl lets it start
// while validate runs.
cudaError_t launch_plan(const Dev& d, const int32_t* req_ids, int B, const int32_t* topk, int32_t* slots,
                        int32_t* hits, int32_t* misses, bool pdl, cudaStream_t st);
cudaError_t launch_gather(const Dev& d, int grid, cudaStream_t st);
// plan + gather fused: each (b, l) CTA copies its own misses right after
// planning them; the last CTA to finish commits the call.
// device_sms: the device's SM count (at most that many units: one CTA per SM
// with more loads in flight per thread).
cudaError_t launch_plan_gather(const Dev& d, const int32_t* req_ids, int B, const int32_t* topk, int32_t* slots,
                               int32_t* hits, int32_t* misses, int device_sms, cudaStream_t st);
cudaError_t prepare_step_kernels(int k, int S, int* gather_grid);

// Attention over assembled slots (tensor cores).
size_t attend_smem_bytes(int k);
// Builds the CUtensorMap (a 128-byte opaque struct, passed as `map`) that
// launch_attend gathers key rows through.
cudaError_t encode_hot_map(const Dev& d, struct CUtensorMap_st* map);
// hot_map: a CUtensorMap over the hot buffer as [R*L*S rows][576] bf16 (box one row x 64, 128B swizzle).
// max_sms: SMs the kernel may occupy (0: all of device_sms, the device's count).
// withhold_keys: the timeout self-test (no key copy is issued, so the kernel's
// bounded waits run out with nothing in flight).
cudaError_t launch_attend(const void* hot_map, const Dev& d, const int32_t* req_ids, int B, const void* q,
                          const int32_t* slots, void* out, float* lse, float sm_scale, int max_sms, int device_sms,
                          cudaStream_t st, bool withhold_keys = false);
// Once per context, on its device: the kernel's shared-memory attribute; *device_sms = the SM count.
cudaError_t prepare_attend(int* device_sms);

// Lifecycle kernels.
cudaError_t launch_reset_request(const Dev& d, int r, int64_t len, int active, cudaStream_t st);
cudaError_t launch_init_lru_all(const Dev& d, cudaStream_t st);
cudaError_t launch_write_back(const Dev& d, const int32_t* req_ids, int n, const void* rows, cudaStream_t st);
cudaError_t launch_extend(const Dev& d, int r, int64_t n, const void* rows, cudaStream_t st);
// Prefetch candidates: per batch entry and layer of the call, the n newest
// tokens of the request, ascending, -1 padded to k ([B][L or 1][k]).
cudaError_t launch_recent_candidates(const Dev& d, const int32_t* req_ids, int B, int n, int32_t* cand, cudaStream_t st);

}  // namespace skv
