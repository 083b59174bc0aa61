// Kernels of one assemble step: validate -> plan (sparse diff + LRU slot
// allocation + map update + slot emission) -> gather (host pool -> HBM).
//
// Pages: per-step, Top-k-driven token-level assembly into a device cache
// ("Sparse Attention-Driven KVCache Management for Domestic AI Supernodes",
// abstract and agenda item 2); the Sparse Diff Kernel moves only the
// difference against the resident set, and the GPU keeps a Top-k LRU buffer
// ("SGLang и Tair представили иерархичную Sparse Attention ...", paragraphs 1
// and 3); the whole step stays graph-executable ("XM-Sparse: Netpreme X-Mem
// ...", section on the SGLang HiSparse integration).
//
// All three kernels have fixed launch shapes that depend only on (B, L, k, S)
// and the device, and read the data-dependent sizes (miss counts, error bits)
// from device memory, so the step can be captured in a CUDA graph.

#include "skv_internal.cuh"

namespace skv {
namespace {

constexpr uint32_t kEmpty = 0xFFFFFFFFu;
constexpr int kMaxIpt = kMaxTopk / kPlanThreads;  // Top-k entries per plan thread

// ---------------------------------------------------------------------------
// Threads that synchronise together: the whole CTA (__syncthreads), or the
// warps [base / 32, (base + n) / 32) on named barrier 1.
// ---------------------------------------------------------------------------
struct CtaSync {
    int n;  // blockDim.x (a multiple of 32)
    static constexpr int base = 0;
    __device__ __forceinline__ void sync() const { __syncthreads(); }
    __device__ __forceinline__ bool any(bool p) const { return __syncthreads_or(p) != 0; }
};
struct WarpGroupSync {
    int n, base;  // multiples of 32
    __device__ __forceinline__ void sync() const { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }
};

// ---------------------------------------------------------------------------
// block-wide exclusive prefix sum over the syncing threads (a multiple of 32,
// <= 1024); `sh` is >= 32 words of shared memory; all of them must call it.
// ---------------------------------------------------------------------------
template <class Sync>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* total, uint32_t* sh, const Sync& sy)
{
    const int rt = (int)threadIdx.x - sy.base;
    const int lane = rt & 31, warp = rt >> 5, nw = sy.n >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    sy.sync();
    if (warp == 0) {
        uint32_t w = lane < nw ? sh[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) sh[lane] = w;
    }
    sy.sync();
    const uint32_t before = warp > 0 ? sh[warp - 1] : 0u;
    *total = sh[nw - 1];
    sy.sync();
    return before + x - v;
}

// block-wide exclusive max over int32 values (identity -1); same calling
// rules as block_excl_scan.
template <class Sync>
__device__ __forceinline__ int32_t block_excl_max(int32_t v, int32_t* sh, const Sync& sy)
{
    const int rt = (int)threadIdx.x - sy.base;
    const int lane = rt & 31, warp = rt >> 5, nw = sy.n >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x = max(x, y);
    }
    int32_t before_in_warp = __shfl_up_sync(0xFFFFFFFFu, x, 1);
    if (lane == 0) before_in_warp = -1;
    if (lane == 31) sh[warp] = x;
    sy.sync();
    if (warp == 0) {
        int32_t w = lane < nw ? sh[lane] : -1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w = max(w, y);
        }
        if (lane < nw) sh[lane] = w;
    }
    sy.sync();
    const int32_t before = warp > 0 ? sh[warp - 1] : -1;
    sy.sync();
    return max(before, before_in_warp);
}

__device__ __forceinline__ bool bit_test(const uint32_t* bm, int s) { return (bm[s >> 5] >> (s & 31)) & 1u; }

// Programmatic dependent launch: the validate kernel lets the plan kernel start
// early; the plan kernel waits for validate's completion (and memory) before
// its first global write.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


// ---------------------------------------------------------------------------
// validate: one CTA per (b, l).  Checks the request id (in range, active, not
// repeated in the batch -- the l == 0 CTA of each b compares with the earlier
// entries) and every Top-k entry (-1 or in [0, len)).  Repeated tokens: a row
// whose non-padding entries are strictly ascending has none (the common case:
// Top-k rows usually come sorted); any other row goes through an
// open-addressing set in shared memory.  Error bits go to CTL_ERR_CALL;
// nothing else is written except the reset of the job-list counter.
// ---------------------------------------------------------------------------
constexpr int kValIpt = kMaxTopk / kValidateThreads;

__global__ void __launch_bounds__(kValidateThreads) validate_kernel(Dev d, const int32_t* __restrict__ req_ids, int B,
                                                                    const int32_t* __restrict__ topk, int table_log2)
{
    extern __shared__ uint32_t table[];
    __shared__ int32_t scan_sh[32];
    __shared__ uint32_t flags;
    pdl_launch_dependents();  // the plan kernel may start its read-only work now
    if (blockIdx.x == 0 && threadIdx.x == 0) d.ctl[CTL_JOBS] = 0;
    if (d.ctl[CTL_ERR] != 0) return;  // sticky error: the call is a no-op
    const int b = d.layer_sel >= 0 ? (int)blockIdx.x : (int)blockIdx.x / d.L;
    const int l = d.layer_sel >= 0 ? d.layer_sel : (int)blockIdx.x % d.L;
    const int32_t r = req_ids[b];
    if (r < 0 || r >= d.R || d.active[r] == 0) {
        if (threadIdx.x == 0) atomicOr(&d.ctl[CTL_ERR_CALL], DEVERR_BAD_REQUEST);
        return;  // uniform across the CTA
    }
    uint32_t f = 0;
    if (d.layer_sel >= 0 || l == 0)  // one CTA per batch entry compares its id with the earlier ones
        for (int j = threadIdx.x; j < b; j += blockDim.x)
            if (req_ids[j] == r) f |= DEVERR_BAD_REQUEST;
    if (threadIdx.x == 0) flags = 0;
    const int64_t len = d.len[r];
    const int k = d.k;
    const int32_t* row = topk + (size_t)blockIdx.x * k;
    // blocked arrangement: thread t holds entries [t*ipt, t*ipt + ipt)
    const int ipt = (k + blockDim.x - 1) / blockDim.x;
    const int i0 = threadIdx.x * ipt;
    int32_t tok[kValIpt];
    int32_t first = -1, prev = -1;
    bool asc = true;
#pragma unroll
    for (int j = 0; j < kValIpt; ++j) {
        tok[j] = -1;
        if (j < ipt && i0 + j < k) {
            const int32_t t = row[i0 + j];
            tok[j] = t;
            if (t == -1) continue;
            if (t < 0 || (int64_t)t >= len) f |= DEVERR_BAD_INDEX;
            if (prev != -1 && t <= prev) asc = false;
            if (t < 0) asc = false;
            if (first == -1) first = t;
            prev = t;
        }
    }
    // the row is strictly ascending iff every segment is and each segment's
    // first entry exceeds the largest entry before it
    const int32_t before = block_excl_max(prev, scan_sh, CtaSync{(int)blockDim.x});
    if (first != -1 && first <= before) asc = false;
    if (!__syncthreads_and(asc)) {
        const int H = 1 << table_log2;
        for (int j = threadIdx.x; j < H; j += blockDim.x) table[j] = kEmpty;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kValIpt; ++j) {
            const int32_t t = tok[j];
            if (j >= ipt || t < 0 || (int64_t)t >= len) continue;  // padding, out of range (already flagged)
            uint32_t h = ((uint32_t)t * 2654435761u) >> (32 - table_log2);
            // H >= 2k, so an empty cell is always reachable: at most H probes
            for (int probe = 0; probe < H; ++probe) {
                const uint32_t p = atomicCAS(&table[h], kEmpty, (uint32_t)t);
                if (p == kEmpty) break;
                if (p == (uint32_t)t) {
                    f |= DEVERR_DUPLICATE;
                    break;
                }
                h = (h + 1) & (uint32_t)(H - 1);
            }
        }
    }
    if (f) atomicOr(&flags, f);
    __syncthreads();
    if (threadIdx.x == 0 && flags) atomicOr(&d.ctl[CTL_ERR_CALL], flags);
}

// ---------------------------------------------------------------------------
// plan: one CTA of kPlanThreads per (b, l).
//   A. sparse diff: probe tok2slot for every entry (blocked arrangement, so a
//      block-wide scan keeps row order); hits mark a bitmap over the slots and
//      are stamped with the new clock; misses are compacted.
//   B. misses are ordered by token (already ordered when the row is sorted;
//      otherwise a bitonic sort in shared memory).
//   C. LRU allocation: walking the unit's LRU order, the first m non-hit
//      slots are the victims, paired in order with the ascending misses.
//   D. new LRU order: untouched slots keep their order, then the slots the
//      step used, by slot index.
//   E. map update per miss (evicted token leaves tok2slot), slot emission,
//      and a gather job (pool row -> hot row).
// ---------------------------------------------------------------------------
struct PlanSmem {
    uint32_t* hitbits;    // [SW]
    uint32_t* vicbits;    // [SW]
    int32_t* out;         // [k]
    unsigned long long* miss;  // [P] (token << 32 | row position)
    uint16_t* victim;     // [k]
    uint16_t* lru_old;    // [S]
    uint16_t* lru_new;    // [S]
};

__host__ __device__ inline int next_pow2(int x)
{
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

__device__ inline PlanSmem carve_plan_smem(uint8_t* base, int k, int S)
{
    PlanSmem m;
    const int SW = (S + 31) / 32;
    size_t o = 0;
    m.miss = (unsigned long long*)(base + o); o += align16((size_t)next_pow2(k) * 8);
    m.hitbits = (uint32_t*)(base + o); o += align16((size_t)SW * 4);
    m.vicbits = (uint32_t*)(base + o); o += align16((size_t)SW * 4);
    m.out = (int32_t*)(base + o); o += align16((size_t)k * 4);
    m.victim = (uint16_t*)(base + o); o += align16((size_t)k * 2);
    m.lru_old = (uint16_t*)(base + o); o += align16((size_t)S * 2);
    m.lru_new = (uint16_t*)(base + o);
    return m;
}

__device__ __forceinline__ int4 ld_stream(const int4* p)
{
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream(int4* p, int4 v)
{
    asm volatile("st.global.cs.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Commit of a call by the last CTA of the fused kernel to finish: every CTA
// has read the clock by then, so it can advance.  All threads of the CTA call
// this.  No CTA waits for another.
__device__ __forceinline__ void finish_call(const Dev& d)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(&d.ctl[CTL_DONE], 1u);
        if (done == gridDim.x - 1) {
            __threadfence();
            const uint32_t e = atomicAdd(&d.ctl[CTL_ERR_CALL], 0u);
            if (atomicAdd(&d.ctl[CTL_ERR], 0u) == 0 && e == 0) {
                d.ctl[CTL_CLOCK] += 1u;
                d.stats[STAT_CALLS] += 1ull;
            }
            d.ctl[CTL_ERR] |= e;
            d.ctl[CTL_ERR_CALL] = 0u;
            d.ctl[CTL_DONE] = 0u;
        }
    }
}

// 16-byte loads each thread keeps in flight in the fused gather: 4 when CTAs
// share SMs (3 per SM; many units keep the link busy together), 8 when every
// unit has an SM to itself (few units: each CTA must cover the link latency
// alone; a bare gather of 16 units x 410 scattered rows took 67 us with 4
// loads in flight a thread and 45 us with 16 or with the rows prefetched into
// L2 first).
constexpr int kFusedUnroll = 4;
constexpr int kFewUnitsUnroll = 8;
// of the 16 warps, those that write the LRU order and the maps beside the
// gather (see plan_kernel).  Measured in one process, steps alternating
// between variants: for few units (128K context, 32 x 4 units: 226.8 us a step
// without the split, 222.7 with 4 warps; 1M context, 4 x 4 units: 60.1 and
// 54.5 us), for the 192 co-resident units of a layer call (16K context, batch
// 192: 3.075 ms a step for eight calls without the split, 3.042 with 2 or 4
// warps); for units in waves it neither costs nor gains (16K context, 192 x 8
// units: 2.932 / 2.925 ms; the same with 40 % fresh tokens: 2.826 / 2.819)
constexpr int kFusedSplitWarps = 2;
constexpr int kFewUnitsSplitWarps = 4;

// kFused = false: the misses become jobs of the global work list, copied by
// gather_kernel.  kFused = true: the CTA copies its own misses (pool row ->
// hot row, 16-byte chunks) right after planning them, so the planning of
// later units overlaps the host-link traffic of earlier ones; each CTA walks
// its own pool region in ascending token order, which keeps the GPU's
// translation of the mapped pool local.
//
// Everything up to the new LRU order (phases A-D) only reads global memory
// and works in shared memory, so it may run before validation has finished:
// indices are bounds-checked against the allocation (not against len) before
// any load, and nothing global is written until pdl_wait() has returned and
// the call is known to be accepted.
//
// UNR: 16-byte loads in flight per thread in the gather; MINB: CTAs per SM the
// register budget is sized for (3 when units run in waves, 1 for few units).
//
// kSplitWarps > 0: as soon as the victims are known (phase C) and the call is
// accepted, the first warps start the gather, and the last kSplitWarps warps
// compute the new LRU order (D) and write the maps and outputs (E) beside it,
// synchronising among themselves on named barrier 1.  The gather needs only
// the sorted misses and their victim slots, and nothing outside this CTA
// reads what D and E write before the call commits.  It pays most where no
// other CTA keeps the link busy while this one plans (every CTA resident).
template <bool kFused, int CPR_CONST, int UNR = kFusedUnroll, int MINB = 3, int kSplitWarps = 0>
__global__ void __launch_bounds__(kPlanThreads, MINB)
    plan_kernel(Dev d, const int32_t* __restrict__ req_ids, const int32_t* __restrict__ topk,
                int32_t* __restrict__ slots_out, int32_t* __restrict__ hits_out, int32_t* __restrict__ misses_out)
{
    static_assert(kSplitWarps == 0 || kFused, "the split gathers: fused kernel only");
    static_assert(kSplitWarps >= 0 && kSplitWarps < kPlanThreads / 32, "some warps must gather");
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ uint32_t scan_sh[32];
    __shared__ uint32_t job_base_sh;
    const int tid = threadIdx.x, NT = (int)blockDim.x;
    const CtaSync sy{NT};
    const int k = d.k, S = d.S;
    const int cpr = CPR_CONST > 0 ? CPR_CONST : d.row_bytes / 16;
    const int32_t* row = topk + (size_t)blockIdx.x * k;
    int32_t* out = slots_out + (size_t)blockIdx.x * k;

    PlanSmem sm = carve_plan_smem(smem_raw, k, S);
    const int b = d.layer_sel >= 0 ? (int)blockIdx.x : (int)blockIdx.x / d.L;
    const int l = d.layer_sel >= 0 ? d.layer_sel : (int)blockIdx.x % d.L;
    const int32_t r = req_ids[b];
    const bool r_ok = r >= 0 && r < d.R;  // uniform over the CTA; validation decides the rest
    const int64_t u = (int64_t)(r_ok ? r : 0) * d.L + l;
    int32_t* t2s = d.tok2slot + u * d.T_max;
    int32_t* s2t = d.slot2tok + u * S;
    uint32_t* tsu = d.ts + u * S;
    uint16_t* lru = d.lru + u * S;
    const int SW = (S + 31) / 32;
    const int ipt = (k + NT - 1) / NT;
    const int i0 = tid * ipt;
    int m = 0, h = 0;

    // D. the slots used by this step go to the back of the LRU order, by slot
    // index (after phase C), by the n threads of `gs`, this one being number rt
    auto new_lru_order = [&](const auto& gs, int rt) {
        const int spt = (S + gs.n - 1) / gs.n;
        const int p0 = rt * spt;
        const int untouched = S - h - m;
        // whole 32-slot words of the bitmaps when the runs tile S in words
        const bool words = (spt & 31) == 0 && spt * gs.n == S;
        uint32_t cnt3 = 0;
        if (words) {
            for (int w = p0 >> 5; w < (p0 + spt) >> 5; ++w) cnt3 += __popc(sm.hitbits[w] | sm.vicbits[w]);
        } else {
            for (int j = 0; j < spt; ++j) {
                const int s = p0 + j;
                if (s < S && (bit_test(sm.hitbits, s) || bit_test(sm.vicbits, s))) ++cnt3;
            }
        }
        uint32_t tot3;
        uint32_t pos = block_excl_scan(cnt3, &tot3, scan_sh, gs);
        if (words) {
            for (int w = p0 >> 5; w < (p0 + spt) >> 5; ++w) {
                for (uint32_t bits = sm.hitbits[w] | sm.vicbits[w]; bits != 0u; bits &= bits - 1u) {
                    const int s = w * 32 + __ffs(bits) - 1;  // ascending within the word
                    if (untouched + (int)pos < S && untouched >= 0) sm.lru_new[untouched + pos++] = (uint16_t)s;
                }
            }
        } else {
            for (int j = 0; j < spt; ++j) {
                const int s = p0 + j;
                if (s < S && (bit_test(sm.hitbits, s) || bit_test(sm.vicbits, s)) && untouched + (int)pos < S &&
                    untouched >= 0)
                    sm.lru_new[untouched + pos++] = (uint16_t)s;
            }
        }
    };

    if (r_ok) {
        for (int w = tid; w < SW; w += NT) {
            sm.hitbits[w] = 0u;
            sm.vicbits[w] = 0u;
        }
        if ((S & 7) == 0) {  // LRU order, 8 slots per 16-byte load
            const uint4* src = reinterpret_cast<const uint4*>(lru);
            uint4* dst = reinterpret_cast<uint4*>(sm.lru_old);
            for (int p = tid; p < S / 8; p += NT) dst[p] = src[p];
        } else {
            for (int p = tid; p < S; p += NT) sm.lru_old[p] = lru[p];
        }

        // A. sparse diff: all row loads, then all (independent) probes; in
        // sm.out a hit holds its slot, a miss -2 (until phase E), padding -1
        int32_t tok[kMaxIpt];
        int32_t hit_slot[kMaxIpt];
#pragma unroll
        for (int j = 0; j < kMaxIpt; ++j) tok[j] = (j < ipt && i0 + j < k) ? row[i0 + j] : -1;
#pragma unroll
        for (int j = 0; j < kMaxIpt; ++j) {
            const int32_t t = tok[j];
            hit_slot[j] = (t >= 0 && (int64_t)t < d.T_max) ? t2s[t] : -1;
        }
        sy.sync();  // bitmaps zeroed, LRU order loaded
        uint32_t missmask = 0, nmiss = 0, nhit = 0;
#pragma unroll
        for (int j = 0; j < kMaxIpt; ++j) {
            const int i = i0 + j;
            if (j >= ipt || i >= k) continue;
            const int32_t t = tok[j], s = hit_slot[j];
            if (t < 0 || (int64_t)t >= d.T_max) {
                sm.out[i] = -1;  // padding (or an invalid entry that validation rejects)
            } else if (s >= 0) {
                sm.out[i] = s;
                atomicOr(&sm.hitbits[s >> 5], 1u << (s & 31));
                ++nhit;
            } else {
                sm.out[i] = -2;
                missmask |= 1u << j;
                ++nmiss;
            }
        }
        uint32_t total;
        const uint32_t excl = block_excl_scan(nmiss | (nhit << 16), &total, scan_sh, sy);
        m = (int)(total & 0xFFFFu);
        h = (int)(total >> 16);
        {
            uint32_t o = excl & 0xFFFFu;
#pragma unroll
            for (int j = 0; j < kMaxIpt; ++j)
                if (missmask & (1u << j))
                    sm.miss[o++] = ((unsigned long long)(uint32_t)tok[j] << 32) | (uint32_t)(i0 + j);
        }
        sy.sync();

        // B. misses in ascending token order
        int unsorted = 0;
        for (int j = tid; j + 1 < m; j += NT)
            if ((sm.miss[j] >> 32) > (sm.miss[j + 1] >> 32)) unsorted = 1;
        if (sy.any(unsorted)) {
            const int P = next_pow2(m);
            for (int j = m + tid; j < P; j += NT) sm.miss[j] = ~0ull;
            sy.sync();
            for (int size = 2; size <= P; size <<= 1) {
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    for (int i = tid; i < P / 2; i += NT) {
                        const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
                        const bool asc = (lo & size) == 0;
                        const unsigned long long a = sm.miss[lo], c = sm.miss[hi];
                        if ((a > c) == asc) {
                            sm.miss[lo] = c;
                            sm.miss[hi] = a;
                        }
                    }
                    sy.sync();
                }
            }
        }

        // C. victims: the first m non-hit slots in LRU order.  Each thread
        // takes a contiguous run of positions, read eight at a time (one
        // 16-byte load) when the runs tile the order exactly.
        const int spt = (S + NT - 1) / NT;
        const int p0 = tid * spt;
        const bool vec = (spt & 7) == 0 && spt * NT == S;
        uint32_t cnt = 0;
        if (vec) {
            for (int j = 0; j < spt; j += 8) {
                const uint4 q = *reinterpret_cast<const uint4*>(sm.lru_old + p0 + j);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) cnt += bit_test(sm.hitbits, (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) ? 0u : 1u;
            }
        } else {
            for (int j = 0; j < spt; ++j) {
                const int p = p0 + j;
                if (p < S && !bit_test(sm.hitbits, sm.lru_old[p])) ++cnt;
            }
        }
        uint32_t tot2;
        uint32_t rank = block_excl_scan(cnt, &tot2, scan_sh, sy);
        auto take = [&](int s) {  // slot s at the next position in LRU order
            if (bit_test(sm.hitbits, s)) return;
            if ((int)rank < m) {
                sm.victim[rank] = (uint16_t)s;
                atomicOr(&sm.vicbits[s >> 5], 1u << (s & 31));
            } else if ((int)rank - m < S) {
                sm.lru_new[rank - m] = (uint16_t)s;
            }
            ++rank;
        };
        if (vec) {
            for (int j = 0; j < spt; j += 8) {
                const uint4 q = *reinterpret_cast<const uint4*>(sm.lru_old + p0 + j);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) take((int)((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu));
            }
        } else {
            for (int j = 0; j < spt; ++j) {
                const int p = p0 + j;
                if (p >= S) break;
                take(sm.lru_old[p]);
            }
        }
        sy.sync();

        if (kSplitWarps == 0) new_lru_order(sy, tid);
    }

    // nothing global has been written yet; from here on the call must be known valid
    pdl_wait();
    if (!r_ok || (d.ctl[CTL_ERR] | d.ctl[CTL_ERR_CALL]) != 0) {  // rejected call: -1 outputs, no state change
        for (int i = tid; i < k; i += NT) out[i] = -1;
        if (tid == 0) {
            hits_out[blockIdx.x] = -1;
            misses_out[blockIdx.x] = -1;
        }
        if (kFused) finish_call(d);
        return;
    }
    const uint32_t now1 = d.ctl[CTL_CLOCK] + 1u;

    // E. stamps, map update and slot emission (plus gather jobs on the job-list
    // path), by the n threads of `gs`, this one being number rt
    auto commit_unit = [&](const auto& gs, int rt) {
        const int n = gs.n;
        for (int i = rt; i < k; i += n) {
            const int32_t s = sm.out[i];
            if (s >= 0) tsu[s] = now1;  // hit
        }
        if (!kFused && rt == 0) job_base_sh = m ? atomicAdd(&d.ctl[CTL_JOBS], (uint32_t)m) : 0u;
        gs.sync();
        for (int j = rt; j < m; j += n) {
            const int v = sm.victim[j];
            const unsigned long long key = sm.miss[j];
            const int32_t t = (int32_t)(key >> 32);
            const int i = (int)(key & 0xFFFFFFFFu);
            const int32_t old = s2t[v];
            if (old >= 0) t2s[old] = -1;
            s2t[v] = t;
            t2s[t] = v;
            tsu[v] = now1;
            sm.out[i] = v;
            if (!kFused) d.jobs[job_base_sh + j] = make_uint2((uint32_t)(u * d.T_max + t), (uint32_t)(u * S + v));
        }
        gs.sync();  // also orders D's writes of the new LRU order before its copy below
        for (int i = rt; i < k; i += n) out[i] = sm.out[i];
        if ((S & 7) == 0) {
            const uint4* src = reinterpret_cast<const uint4*>(sm.lru_new);
            uint4* dst = reinterpret_cast<uint4*>(lru);
            for (int p = rt; p < S / 8; p += n) dst[p] = src[p];
        } else {
            for (int p = rt; p < S; p += n) lru[p] = sm.lru_new[p];
        }
        if (rt == 0) {
            hits_out[blockIdx.x] = h;
            misses_out[blockIdx.x] = m;
            if (h) atomicAdd(&d.stats[STAT_HITS], (unsigned long long)h);
            if (kFused && m) atomicAdd(&d.stats[STAT_MISSES], (unsigned long long)m);
        }
    };

    // F. gather: pool row (u, token) -> hot row (u, victim slot), by n threads
    auto gather = [&](int rt, int n) {
        const int4* __restrict__ src = reinterpret_cast<const int4*>(d.pool) + (size_t)u * d.T_max * cpr;
        int4* __restrict__ dst = reinterpret_cast<int4*>(d.hot) + (size_t)u * S * cpr;
        const int chunks = m * cpr;
        for (int base = rt; base < chunks; base += n * UNR) {
            int4 v[UNR];
            uint32_t o[UNR];  // victim * cpr + w < S * cpr <= 2^14 * 2^12
#pragma unroll
            for (int j = 0; j < UNR; ++j) {
                const int c = base + j * n;
                if (c < chunks) {
                    const int jj = c / cpr;
                    const int w = c - jj * cpr;
                    const int32_t t = (int32_t)(sm.miss[jj] >> 32);
                    o[j] = (uint32_t)sm.victim[jj] * (uint32_t)cpr + (uint32_t)w;
                    v[j] = ld_stream(src + (size_t)t * cpr + w);
                }
            }
#pragma unroll
            for (int j = 0; j < UNR; ++j)
                if (base + j * n < chunks) st_stream(dst + o[j], v[j]);
        }
    };

    if (kSplitWarps > 0) {
        constexpr int kGatherThreads = kPlanThreads - 32 * kSplitWarps;
        if (tid < kGatherThreads) {
            gather(tid, kGatherThreads);
        } else {
            const WarpGroupSync gs{NT - kGatherThreads, kGatherThreads};
            new_lru_order(gs, tid - kGatherThreads);
            commit_unit(gs, tid - kGatherThreads);
        }
    } else {
        commit_unit(sy, tid);
        if (kFused) gather(tid, NT);
    }
    if (kFused) finish_call(d);
}

// ---------------------------------------------------------------------------
// gather: copy every queued row (pool row -> hot row) in 16-byte chunks.
// The chunk space (jobs x chunks per row) is walked grid-stride; each thread
// issues U independent 16-byte loads from the mapped host pool before it
// stores them, to keep many host-link reads in flight.  Block 0 also commits
// the call: clock + 1 and statistics on success, error bits into the sticky
// word.
// ---------------------------------------------------------------------------
template <int CPR_CONST, int U>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(Dev d, int cpr_rt)
{
    const int cpr = CPR_CONST > 0 ? CPR_CONST : cpr_rt;  // 16-byte chunks per row
    const uint32_t M = d.ctl[CTL_JOBS];
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const uint32_t e = d.ctl[CTL_ERR_CALL];
        if (d.ctl[CTL_ERR] == 0 && e == 0) {
            d.ctl[CTL_CLOCK] += 1u;
            d.stats[STAT_CALLS] += 1ull;
            d.stats[STAT_MISSES] += (unsigned long long)M;
        }
        d.ctl[CTL_ERR] |= e;
        d.ctl[CTL_ERR_CALL] = 0u;
    }
    const uint64_t total = (uint64_t)M * (uint64_t)cpr;
    const int4* __restrict__ src = reinterpret_cast<const int4*>(d.pool);
    int4* __restrict__ dst = reinterpret_cast<int4*>(d.hot);
    const uint2* __restrict__ jobs = d.jobs;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x * U;
    for (uint64_t base = (uint64_t)blockIdx.x * blockDim.x * U + threadIdx.x; base < total; base += stride) {
        int4 v[U];
        uint64_t o[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const uint64_t c = base + (uint64_t)j * blockDim.x;
            if (c < total) {
                const uint32_t job = (uint32_t)(c / (uint64_t)cpr);
                const uint32_t w = (uint32_t)(c - (uint64_t)job * cpr);
                const uint2 jb = jobs[job];
                o[j] = (uint64_t)jb.y * cpr + w;
                v[j] = ld_stream(src + (uint64_t)jb.x * cpr + w);
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const uint64_t c = base + (uint64_t)j * blockDim.x;
            if (c < total) st_stream(dst + o[j], v[j]);
        }
    }
}

constexpr int kGatherUnroll = 4;

}  // namespace

size_t plan_smem_bytes(int k, int S)
{
    const int SW = (S + 31) / 32;
    return align16((size_t)next_pow2(k) * 8) + 2 * align16((size_t)SW * 4) + align16((size_t)k * 4) +
           align16((size_t)k * 2) + 2 * align16((size_t)S * 2);
}

static int table_log2_for(int k)
{
    int lg = 1;
    while ((1 << lg) < 2 * k) ++lg;
    return lg;
}

size_t validate_smem_bytes(int k) { return ((size_t)1 << table_log2_for(k)) * 4; }

cudaError_t prepare_step_kernels(int k, int S, int* gather_grid)
{
    // the attributes are per function, not per context: allow the largest
    // (k, S) any context may use, so contexts of different shapes coexist
    (void)k;
    (void)S;
    const int plan_max = (int)plan_smem_bytes(kMaxTopk, kMaxSlots);
    cudaError_t e = cudaFuncSetAttribute(plan_kernel<false, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, plan_max);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(plan_kernel<true, 72, kFusedUnroll, 3, kFusedSplitWarps>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, plan_max);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(plan_kernel<true, 0, kFusedUnroll, 3, kFusedSplitWarps>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, plan_max);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(plan_kernel<true, 72, kFewUnitsUnroll, 1, kFewUnitsSplitWarps>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, plan_max);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(plan_kernel<true, 0, kFewUnitsUnroll, 1, kFewUnitsSplitWarps>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, plan_max);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(validate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)validate_smem_bytes(kMaxTopk));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_kernel<72, kGatherUnroll>,
                                                           kGatherThreads, 0)) != cudaSuccess)
        return e;
    // every kernel of the step is loaded here, at context creation (CUDA loads
    // functions lazily), so that no assemble call loads code later
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, gather_kernel<0, kGatherUnroll>)) != cudaSuccess) return e;
    *gather_grid = sms * (per_sm > 0 ? per_sm : 1);
    return cudaSuccess;
}

cudaError_t launch_validate(const Dev& d, const int32_t* req_ids, int B, const int32_t* topk, cudaStream_t st)
{
    const int lg = table_log2_for(d.k);
    validate_kernel<<<call_units(d, B), kValidateThreads, validate_smem_bytes(d.k), st>>>(d, req_ids, B, topk, lg);
    return cudaGetLastError();
}

cudaError_t launch_plan(const Dev& d, const int32_t* req_ids, int B, const int32_t* topk, int32_t* slots,
                        int32_t* hits, int32_t* misses, bool pdl, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(call_units(d, B));
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = plan_smem_bytes(d.k, d.S);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, plan_kernel<false, 0>, d, req_ids, topk, slots, hits, misses);
}

cudaError_t launch_plan_gather(const Dev& d, const int32_t* req_ids, int B, const int32_t* topk, int32_t* slots,
                               int32_t* hits, int32_t* misses, int device_sms, cudaStream_t st)
{
    // few units (at most one per SM): the variant with more loads in flight
    // per thread, each CTA alone on its SM.  No variant prefetches the missing
    // rows into L2 ahead of the gather: measured -1.5 % to -4 % for units in
    // waves, 3.22 against 3.12 ms a step for eight layer calls of 192
    // co-resident units, and for few units (a warp of its own issuing the
    // prefetches while the CTA planned) 231.6 against 227.5 us a step at 128K
    // context (32 x 4 units) and 60.0 against 60.1 us at 1M (4 x 4 units).
    const int grid = call_units(d, B);
    const bool few = grid <= device_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = plan_smem_bytes(d.k, d.S);
    cfg.stream = st;
    // Programmatic dependent launch (planning overlaps validation) only for
    // few units, at most one CTA per SM: measured 55 us from validation's
    // start to the commit with it, 62 us without, for 16 units.  With more
    // units it costs time: 3.016 ms a step with it and 2.947 ms without for
    // 1536 units in waves, and 3.61 ms against 3.25 ms for eight calls of 192
    // (co-resident, three CTAs to an SM).
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = few ? 1 : 0;
    if (d.row_bytes == 1152)
        return few ? cudaLaunchKernelEx(&cfg, plan_kernel<true, 72, kFewUnitsUnroll, 1, kFewUnitsSplitWarps>, d,
                                        req_ids, topk, slots, hits, misses)
                   : cudaLaunchKernelEx(&cfg, plan_kernel<true, 72, kFusedUnroll, 3, kFusedSplitWarps>, d, req_ids,
                                        topk, slots, hits, misses);
    return few ? cudaLaunchKernelEx(&cfg, plan_kernel<true, 0, kFewUnitsUnroll, 1, kFewUnitsSplitWarps>, d, req_ids,
                                    topk, slots, hits, misses)
               : cudaLaunchKernelEx(&cfg, plan_kernel<true, 0, kFusedUnroll, 3, kFusedSplitWarps>, d, req_ids, topk,
                                    slots, hits, misses);
}

cudaError_t launch_gather(const Dev& d, int grid, cudaStream_t st)
{
    const int cpr = d.row_bytes / 16;
    if (cpr == 72)
        gather_kernel<72, kGatherUnroll><<<grid, kGatherThreads, 0, st>>>(d, cpr);
    else
        gather_kernel<0, kGatherUnroll><<<grid, kGatherThreads, 0, st>>>(d, cpr);
    return cudaGetLastError();
}

}  // namespace skv
