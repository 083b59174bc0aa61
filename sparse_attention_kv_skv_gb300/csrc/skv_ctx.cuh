// The context object behind the opaque skv_ctx handle (internal; not ABI).
#pragma once

#include <vector>

#include <cuda.h>

#include "skv.h"
#include "skv_internal.cuh"

struct skv_ctx {
    skv_config cfg{};
    skv::Dev d{};
    uint8_t* pool_host = nullptr;  // same memory as d.pool (mapped)
    std::vector<uint8_t> active_h;  // host mirror of the request table
    int32_t* st_req = nullptr;      // staging for skv_assemble_host
    int32_t* st_topk = nullptr;
    int32_t* st_slots = nullptr;
    int32_t* st_hits = nullptr;
    int32_t* st_misses = nullptr;
    uint32_t* host_word = nullptr;  // pinned word for reading the error bits
    cudaEvent_t ev_before = nullptr, ev_after = nullptr;
    int gather_grid = 0;
    CUtensorMap hot_map{};  // TMA view of the hot buffer for the attention consumer (built on first use)
    bool hot_map_ready = false;
    int attend_sms = 0;     // SMs the attention kernel may occupy (0: all)
    int device_sms = 0;     // SMs of the context's device
    int pool_node_wanted = -1;   // host NUMA node the pool was asked to live on (-1: none)
    int pool_node_seen = -1;     // node holding most sampled pool pages (-1: not reported)
    float pool_node_frac = 0.0f; // share of the sampled pages on pool_node_seen
};

namespace skv {
// Sets the message returned by skv_last_cuda_error on this thread.
void set_last_error_message(const char* msg);
// Loads skv_assemble_noalloc's static work list on `device` (current) and
// caches its address, so that no later call loads or allocates anything.
cudaError_t noalloc_prepare(int device);
}  // namespace skv
