// CPU ORACLE for the sparse KV assembly path -- TEST INFRASTRUCTURE ONLY.
//
// Only the test suite, the package smoke check and the benchmark's CPU
// baseline may load this library.  The product (the CUDA library and its
// Python binding) never calls it and shares no code with it: no headers, no
// helpers, no tables.  The two meet only in the seeded inputs.
//
// What it computes, and where the pages state it:
//
// * Host storage: the full KV history of every request lives in a host memory
//   pool; the device keeps only a cache of hot tokens ("Sparse
//   Attention-Driven KVCache Management for Domestic AI Supernodes", abstract
//   and agenda item 2: host storage, device cache, index mapping; "SGLang и
//   Tair представили иерархичную Sparse Attention ...", paragraph 1: full KV in
//   the CPU tier, a Top-k LRU buffer on the GPU).
// * Per decode step and per (request, layer), the Top-k token indices decide
//   which tokens must be on the device; only the difference against what is
//   already resident is moved ("SGLang и Tair ...", paragraph 3: incremental
//   transfer of sparse changes through the Sparse Diff Kernel; KVCache
//   Management talk, abstract: token-level, on-demand assembly of the data the
//   current computation needs).
// * Room for missing tokens is made by least-recently-used replacement in the
//   device buffer ("SGLang и Tair ...", paragraph 1, the Top-k LRU buffer).
// * The attention kernel receives a fixed-shape tensor of slot indices, which
//   keeps the step graph-executable (KVCache Management talk, abstract and
//   agenda item 2, the UniDex index-copy operator; "XM-Sparse ...", section on
//   the SGLang HiSparse integration: CUDA Graph support).
// * Calls follow the request lifecycle publish / acquire / write back /
//   release ("XM-Sparse ...", same section).
//
// The pages are silent on the exact replacement order.  The readings taken
// here: one hot buffer of S slots per (request, layer); a global step clock
// that advances once per successful assemble; every slot used by the step's
// Top-k (hits and newly filled) gets the new clock value; victims are the m
// slots with the smallest (last-use step, slot index) among slots not hit in
// this step; the missing tokens, in ascending token order, take the victims in
// that order.  A rejected call changes nothing.
//
// State per (request, layer) follows the plainest data structures for that
// reading: a hash map token -> slot, arrays slot -> token and slot -> last-use
// step, and a doubly linked list of all slots kept in LRU order (front = least
// recently used, ties by slot index).  Gathers are memcpy.  Nothing is blocked,
// fused or reordered; the only parallelism is an optional OpenMP loop over the
// independent (request, layer) units of one step.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <list>
#include <unordered_map>
#include <unordered_set>
#include <utility>
#include <vector>

namespace {

// error bits of the sticky error word (same meaning as the library's)
constexpr int32_t E_BAD_REQUEST = 1;   // request id out of range, inactive, or repeated in one call
constexpr int32_t E_BAD_INDEX = 2;     // Top-k entry outside [0, len) and not -1
constexpr int32_t E_DUPLICATE = 4;     // a token appears twice in one (request, layer) row
constexpr int32_t E_CONTEXT_FULL = 8;  // write_back on a request whose pool region is full

struct Unit {
    std::unordered_map<int32_t, int32_t> tok2slot;  // resident token -> slot
    std::vector<int32_t> slot2tok;                  // slot -> token, -1 = empty
    std::vector<uint32_t> ts;                       // slot -> step of last use, 0 = never
    std::list<int32_t> lru;                         // all S slots, least recently used first
    std::vector<uint8_t> hot;                       // device-cache contents [S][row_bytes]
    std::unordered_map<int64_t, std::vector<uint8_t>> appended;  // rows added by write_back, by position
};

struct Request {
    bool active = false;
    int64_t len = 0;       // tokens in the pool (published + appended)
    int64_t base_len = 0;  // tokens that were published (read from the pool view)
    std::vector<Unit> units;  // one per layer
};

struct Oracle {
    int32_t R, L, k, S, row_bytes;
    int64_t T_max;
    const uint8_t* pool;  // read-only view [R][L][T_max][row_bytes] of the published rows
    std::vector<Request> req;
    uint32_t now = 0;
    int32_t err = 0;
};

void reset_request(Oracle* o, Request& q)
{
    q.units.clear();
    q.units.resize(o->L);
    for (Unit& u : q.units) {
        u.slot2tok.assign(o->S, -1);
        u.ts.assign(o->S, 0);
        for (int32_t s = 0; s < o->S; ++s) u.lru.push_back(s);
        u.hot.assign((size_t)o->S * o->row_bytes, 0);
    }
}

const uint8_t* pool_row(const Oracle* o, const Request& q, const Unit& u, int32_t r, int32_t l, int64_t t)
{
    if (t < q.base_len) return o->pool + (((size_t)r * o->L + l) * o->T_max + t) * o->row_bytes;
    return u.appended.at(t).data();
}

// One (request, layer) unit of one assemble step.  `row` holds k Top-k
// entries; the k slot indices go to `out`.
void assemble_unit(Oracle* o, int32_t r, int32_t l, const int32_t* row, int32_t* out, int32_t* n_hit,
                   int32_t* n_miss, uint32_t now)
{
    Request& q = o->req[r];
    Unit& u = q.units[l];
    std::vector<int32_t> hit_slots;
    std::vector<std::pair<int32_t, int32_t>> missing;  // (token, position in the row)
    // sparse diff: resident tokens are hits, the rest are misses
    for (int32_t i = 0; i < o->k; ++i) {
        const int32_t t = row[i];
        if (t == -1) {
            out[i] = -1;
            continue;
        }
        auto it = u.tok2slot.find(t);
        if (it != u.tok2slot.end()) {
            out[i] = it->second;
            hit_slots.push_back(it->second);
        } else {
            missing.emplace_back(t, i);
        }
    }
    // a slot hit in this step is never a victim: take hits out of the LRU list
    std::unordered_set<int32_t> hit_set(hit_slots.begin(), hit_slots.end());
    u.lru.remove_if([&](int32_t s) { return hit_set.count(s) != 0; });
    // misses in ascending token order take the least recently used slots in order
    std::sort(missing.begin(), missing.end());
    const int32_t m = (int32_t)missing.size();
    std::vector<int32_t> victims;
    for (int32_t j = 0; j < m; ++j) {
        victims.push_back(u.lru.front());
        u.lru.pop_front();
    }
    for (int32_t j = 0; j < m; ++j) {
        const int32_t v = victims[j];
        const int32_t t = missing[j].first;
        const int32_t old = u.slot2tok[v];
        if (old >= 0) u.tok2slot.erase(old);
        u.slot2tok[v] = t;
        u.tok2slot[t] = v;
        std::memcpy(u.hot.data() + (size_t)v * o->row_bytes, pool_row(o, q, u, r, l, t), o->row_bytes);
        out[missing[j].second] = v;
    }
    // every slot the step used becomes most recently used, in slot order
    std::vector<int32_t> touched(hit_slots);
    touched.insert(touched.end(), victims.begin(), victims.end());
    std::sort(touched.begin(), touched.end());
    for (int32_t s : touched) {
        u.ts[s] = now;
        u.lru.push_back(s);
    }
    *n_hit = (int32_t)hit_slots.size();
    *n_miss = m;
}

}  // namespace

extern "C" {

void* orc_create(int32_t R, int32_t L, int64_t T_max, int32_t row_bytes, int32_t k, int32_t S,
                 const uint8_t* pool)
{
    if (R < 1 || L < 1 || T_max < 1 || row_bytes < 1 || k < 1 || S < k || !pool) return nullptr;
    Oracle* o = new Oracle();
    o->R = R; o->L = L; o->T_max = T_max; o->row_bytes = row_bytes; o->k = k; o->S = S; o->pool = pool;
    o->req.resize(R);
    return o;
}

void orc_destroy(void* h) { delete static_cast<Oracle*>(h); }

// Returns the new request id (lowest free id), -1 if none is free, -2 if T is
// out of range.  Rows [0, T) of the request must be in the pool view before
// the first assemble that reads them.
int32_t orc_publish(void* h, int64_t T)
{
    Oracle* o = static_cast<Oracle*>(h);
    if (T < 0 || T > o->T_max) return -2;
    for (int32_t r = 0; r < o->R; ++r) {
        Request& q = o->req[r];
        if (q.active) continue;
        q.active = true;
        q.len = T;
        q.base_len = T;
        reset_request(o, q);
        return r;
    }
    return -1;
}

// 0 on success, -1 if r is not an active request.
int32_t orc_release(void* h, int32_t r)
{
    Oracle* o = static_cast<Oracle*>(h);
    if (r < 0 || r >= o->R || !o->req[r].active) return -1;
    Request& q = o->req[r];
    q.active = false;
    q.len = 0;
    q.base_len = 0;
    q.units.clear();
    return 0;
}

// Append one row per layer to each listed request.  rows is [n][L][row_bytes].
// Returns the error bits of this call (0 on success); a rejected call changes
// nothing except the sticky error word.
int32_t orc_write_back(void* h, const int32_t* req_ids, int32_t n, const uint8_t* rows)
{
    Oracle* o = static_cast<Oracle*>(h);
    if (n <= 0) return 0;
    if (o->err) return o->err;
    int32_t e = 0;
    std::unordered_set<int32_t> seen;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t r = req_ids[i];
        if (r < 0 || r >= o->R || !o->req[r].active || !seen.insert(r).second) {
            e |= E_BAD_REQUEST;
            continue;
        }
        if (o->req[r].len >= o->T_max) e |= E_CONTEXT_FULL;
    }
    if (e) {
        o->err |= e;
        return e;
    }
    for (int32_t i = 0; i < n; ++i) {
        Request& q = o->req[req_ids[i]];
        for (int32_t l = 0; l < o->L; ++l) {
            const uint8_t* src = rows + ((size_t)i * o->L + l) * o->row_bytes;
            q.units[l].appended[q.len] = std::vector<uint8_t>(src, src + o->row_bytes);
        }
        q.len += 1;
    }
    return 0;
}

// One decode step over the units of `layers` (all L layers when layer < 0,
// else only that layer): topk is [B][nl][k] with nl = L or 1; slots (same
// shape) receives slot indices (-1 for -1 entries); hits / misses are
// [B][nl].  Returns the error bits of this call, or the already-set sticky
// word; on any error the outputs are -1 and nothing else changes.
static int32_t assemble_units(Oracle* o, const int32_t* req_ids, int32_t B, int32_t layer, const int32_t* topk,
                              int32_t* slots, int32_t* hits, int32_t* misses, int32_t nthreads)
{
    const int64_t nl = layer < 0 ? o->L : 1, k = o->k;
    if (B <= 0) return 0;
    auto reject = [&]() {
        std::fill(slots, slots + (size_t)B * nl * k, -1);
        std::fill(hits, hits + (size_t)B * nl, -1);
        std::fill(misses, misses + (size_t)B * nl, -1);
    };
    if (o->err) {
        reject();
        return o->err;
    }
    // validate everything before changing anything
    int32_t e = 0;
    std::unordered_set<int32_t> seen;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t r = req_ids[b];
        if (r < 0 || r >= o->R || !o->req[r].active) {
            e |= E_BAD_REQUEST;
            continue;
        }
        if (!seen.insert(r).second) e |= E_BAD_REQUEST;
        const int64_t len = o->req[r].len;
        for (int64_t j = 0; j < nl; ++j) {
            std::unordered_set<int32_t> row_tokens;
            const int32_t* row = topk + ((size_t)b * nl + j) * k;
            for (int64_t i = 0; i < k; ++i) {
                const int32_t t = row[i];
                if (t == -1) continue;
                if (t < 0 || t >= len) e |= E_BAD_INDEX;
                else if (!row_tokens.insert(t).second) e |= E_DUPLICATE;
            }
        }
    }
    if (e) {
        o->err |= e;
        reject();
        return e;
    }
    const uint32_t now = o->now + 1;
    const int64_t units = (int64_t)B * nl;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t x = 0; x < units; ++x) {
        const int32_t b = (int32_t)(x / nl);
        const int32_t l = layer < 0 ? (int32_t)(x % nl) : layer;
        assemble_unit(o, req_ids[b], l, topk + x * k, slots + x * k, hits + x, misses + x, now);
    }
    o->now = now;
    return 0;
}

// One decode step over all layers: topk is [B][L][k].
int32_t orc_assemble(void* h, const int32_t* req_ids, int32_t B, const int32_t* topk, int32_t* slots,
                     int32_t* hits, int32_t* misses, int32_t nthreads)
{
    return assemble_units(static_cast<Oracle*>(h), req_ids, B, -1, topk, slots, hits, misses, nthreads);
}

// One step of one layer: topk is [B][k]; the clock advances by one as for a
// full step, so the replacement order of a (request, layer) follows the order
// of the calls that touched it.  Returns -100 for a layer outside [0, L).
int32_t orc_assemble_layer(void* h, const int32_t* req_ids, int32_t B, int32_t layer, const int32_t* topk,
                           int32_t* slots, int32_t* hits, int32_t* misses, int32_t nthreads)
{
    Oracle* o = static_cast<Oracle*>(h);
    if (layer < 0 || layer >= o->L) return -100;
    return assemble_units(o, req_ids, B, layer, topk, slots, hits, misses, nthreads);
}

// Append n rows per layer to request r: rows is [L][n][row_bytes].  Returns
// the error bits (0 on success; the sticky word if already set), or -1 if r
// is not an active request (nothing changes).
int32_t orc_extend(void* h, int32_t r, const uint8_t* rows, int64_t n)
{
    Oracle* o = static_cast<Oracle*>(h);
    if (r < 0 || r >= o->R || !o->req[r].active) return -1;
    if (n <= 0) return 0;
    if (o->err) return o->err;
    Request& q = o->req[r];
    if (q.len + n > o->T_max) {
        o->err |= E_CONTEXT_FULL;
        return E_CONTEXT_FULL;
    }
    for (int32_t l = 0; l < o->L; ++l)
        for (int64_t j = 0; j < n; ++j) {
            const uint8_t* src = rows + ((size_t)l * n + j) * o->row_bytes;
            q.units[l].appended[q.len + j] = std::vector<uint8_t>(src, src + o->row_bytes);
        }
    q.len += n;
    return 0;
}

// Read and clear the sticky error word.
int32_t orc_get_error(void* h)
{
    Oracle* o = static_cast<Oracle*>(h);
    const int32_t e = o->err;
    o->err = 0;
    return e;
}

uint32_t orc_now(void* h) { return static_cast<Oracle*>(h)->now; }

// Export one request's state.  Any pointer may be null.  slot2tok, ts and lru
// are [L][S] (lru lists slots least recently used first); tok2slot is
// [L][T_max] (-1 = not resident).  For an inactive request the arrays are
// filled with their empty values and len = 0.
void orc_export(void* h, int32_t r, int32_t* slot2tok, uint32_t* ts, int32_t* tok2slot, int32_t* lru,
                int64_t* len, int32_t* active)
{
    Oracle* o = static_cast<Oracle*>(h);
    const Request& q = o->req[r];
    if (len) *len = q.len;
    if (active) *active = q.active ? 1 : 0;
    for (int32_t l = 0; l < o->L; ++l) {
        const size_t so = (size_t)l * o->S;
        if (!q.active) {
            if (slot2tok) std::fill(slot2tok + so, slot2tok + so + o->S, -1);
            if (ts) std::fill(ts + so, ts + so + o->S, 0u);
            if (lru) for (int32_t s = 0; s < o->S; ++s) lru[so + s] = s;
            if (tok2slot) std::fill(tok2slot + (size_t)l * o->T_max, tok2slot + (size_t)(l + 1) * o->T_max, -1);
            continue;
        }
        const Unit& u = q.units[l];
        if (slot2tok) std::copy(u.slot2tok.begin(), u.slot2tok.end(), slot2tok + so);
        if (ts) std::copy(u.ts.begin(), u.ts.end(), ts + so);
        if (lru) std::copy(u.lru.begin(), u.lru.end(), lru + so);
        if (tok2slot) {
            int32_t* d = tok2slot + (size_t)l * o->T_max;
            std::fill(d, d + o->T_max, -1);
            for (const auto& kv : u.tok2slot) d[kv.first] = kv.second;
        }
    }
}

// Copy one request's device-cache contents [L][S][row_bytes] (zeros if inactive).
void orc_export_hot(void* h, int32_t r, uint8_t* dst)
{
    Oracle* o = static_cast<Oracle*>(h);
    const Request& q = o->req[r];
    const size_t per = (size_t)o->S * o->row_bytes;
    for (int32_t l = 0; l < o->L; ++l) {
        if (q.active) std::memcpy(dst + l * per, q.units[l].hot.data(), per);
        else std::memset(dst + l * per, 0, per);
    }
}

// The pool row (r, l, t) as the oracle sees it (published or appended).
// Returns 0, or -1 if the row does not exist.
int32_t orc_pool_row(void* h, int32_t r, int32_t l, int64_t t, uint8_t* dst)
{
    Oracle* o = static_cast<Oracle*>(h);
    if (r < 0 || r >= o->R || !o->req[r].active || l < 0 || l >= o->L || t < 0 || t >= o->req[r].len) return -1;
    const Request& q = o->req[r];
    std::memcpy(dst, pool_row(o, q, q.units[l], r, l, t), o->row_bytes);
    return 0;
}

}  // extern "C"
