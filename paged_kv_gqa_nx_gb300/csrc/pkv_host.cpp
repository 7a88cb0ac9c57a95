// pkv_host.cpp -- host core and C ABI of libpkv.
//
// Host side of the paged KV cache: the refcounted block pool (LIFO free
// stack, refcounts), sequences with their page tables, ensure_append with
// copy-on-append, advance, fork, truncate; and the per-layer calls that build
// one descriptor blob per call (page-table changes, batch rows, append rows,
// split-K work units, merge items), upload it through a pinned staging ring
// and launch the kernels on the pool stream.
//
// Call contract: "nx_f32_attn_paged.nx source" (header comment: ensure_append
// once per step, append + attend per layer, advance once after all layers);
// pool behaviour: "nx_paged_kv_gate.nx source" (KAT, FORK, REWIND sections).
#include "../../include/pkv.h"
#include "pkv_internal.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <list>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

using namespace pkv;

// ------------------------------------------------------------------ state ----
namespace {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::atomic<int32_t> g_split_keys{1024};
std::atomic<int32_t> g_fused_append{1};
std::atomic<int32_t> g_cascade{1};
std::atomic<int32_t> g_prefill_pairing{2};
std::atomic<int64_t> g_launches{0};

// Optional per-launch CUDA-event timing.
struct Profiler {
    std::mutex mu;
    bool on = false;
    struct Rec {
        int kind;
        cudaEvent_t a, b;
    };
    std::vector<Rec> recs;
    std::vector<cudaEvent_t> spare;
    double ms[PKV_KERNEL_KINDS] = {};
    int64_t n[PKV_KERNEL_KINDS] = {};

    cudaEvent_t get() {
        if (!spare.empty()) {
            cudaEvent_t e = spare.back();
            spare.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
    // Fold finished records into the totals (caller holds mu).
    void drain() {
        for (auto &r : recs) {
            cudaEventSynchronize(r.b);
            float t = 0.f;
            if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
                ms[r.kind] += t;
                n[r.kind] += 1;
            }
            spare.push_back(r.a);
            spare.push_back(r.b);
        }
        recs.clear();
    }
};
Profiler g_prof;

// Enqueue one kernel through `f`, counting it and (when profiling) timing it.
template <class F>
cudaError_t launch(int kind, cudaStream_t s, F &&f) {
    cudaEvent_t a = nullptr, b = nullptr;
    bool on;
    {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        on = g_prof.on;
        if (on) {
            a = g_prof.get();
            b = g_prof.get();
        }
    }
    if (on) cudaEventRecord(a, s);
    cudaError_t e = f();
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (on) {
        cudaEventRecord(b, s);
        std::lock_guard<std::mutex> lk(g_prof.mu);
        g_prof.recs.push_back({kind, a, b});
    }
    return e;
}

// The library's stream-ordered memory pool, one per device; memory is kept
// (release threshold = max) so steady-state calls reuse it without the OS.
std::mutex g_mempool_mu;
cudaMemPool_t g_mempool[64] = {};

cudaError_t mempool_for(int dev, cudaMemPool_t *out) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mempool_mu);
    if (!g_mempool[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t mp = nullptr;
        cudaError_t e = cudaMemPoolCreate(&mp, &props);
        if (e != cudaSuccess) return e;
        uint64_t thr = ~0ull;
        cudaMemPoolSetAttribute(mp, cudaMemPoolAttrReleaseThreshold, &thr);
        g_mempool[dev] = mp;
    }
    *out = g_mempool[dev];
    return cudaSuccess;
}

// Growable stream-ordered device buffer.
struct DevBuf {
    void *p = nullptr;
    size_t cap = 0;
    cudaError_t ensure(size_t n, cudaStream_t s, int dev) {
        if (n <= cap) return cudaSuccess;
        cudaMemPool_t mp;
        cudaError_t e = mempool_for(dev, &mp);
        if (e != cudaSuccess) return e;
        if (p) cudaFreeAsync(p, s);
        p = nullptr;
        cap = 0;
        size_t nc = std::max<size_t>(n, 4096);
        e = cudaMallocFromPoolAsync(&p, nc, mp, s);
        if (e != cudaSuccess) {
            p = nullptr;
            return e;
        }
        cap = nc;
        return cudaSuccess;
    }
    void release(cudaStream_t s) {
        if (p) cudaFreeAsync(p, s);
        p = nullptr;
        cap = 0;
    }
};

// Pinned staging ring for host->device descriptor uploads.  A slot is reused
// only after the copy that last read it has completed.
struct Stager {
    static constexpr int N = 8;
    struct Slot {
        void *h = nullptr;
        size_t cap = 0;
        cudaEvent_t ev = nullptr;
        bool pending = false;
    };
    Slot slots[N];
    int next = 0;

    cudaError_t upload(void *dst, const void *src, size_t n, cudaStream_t s) {
        Slot &sl = slots[next];
        next = (next + 1) % N;
        if (sl.pending) {
            cudaEventSynchronize(sl.ev);
            sl.pending = false;
        }
        if (sl.cap < n) {
            if (sl.h) cudaFreeHost(sl.h);
            sl.h = nullptr;
            sl.cap = 0;
            size_t nc = std::max<size_t>(n, 64 * 1024);
            cudaError_t e = cudaMallocHost(&sl.h, nc);
            if (e != cudaSuccess) return e;
            sl.cap = nc;
        }
        if (!sl.ev) {
            cudaError_t e = cudaEventCreateWithFlags(&sl.ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        std::memcpy(sl.h, src, n);
        cudaError_t e = cudaMemcpyAsync(dst, sl.h, n, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return e;
        e = cudaEventRecord(sl.ev, s);
        if (e != cudaSuccess) return e;
        sl.pending = true;
        return cudaSuccess;
    }
    void destroy() {
        for (auto &sl : slots) {
            if (sl.pending) cudaEventSynchronize(sl.ev);
            if (sl.ev) cudaEventDestroy(sl.ev);
            if (sl.h) cudaFreeHost(sl.h);
            sl = Slot{};
        }
    }
};

// Host-side descriptor blob; sections start on 16-byte boundaries.
struct Blob {
    std::vector<unsigned char> b;
    void clear() { b.clear(); }
    template <class T>
    size_t put(const T *data, size_t count) {
        size_t off = (b.size() + 15) & ~static_cast<size_t>(15);
        b.resize(off + count * sizeof(T));
        if (count) std::memcpy(b.data() + off, data, count * sizeof(T));
        return off;
    }
    size_t size() const { return std::max<size_t>(b.size(), 16); }
};

struct DevGuard {
    int prev = -1;
    explicit DevGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    }
    ~DevGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

}  // namespace

// ------------------------------------------------------------- pool, seq ----

struct pkv_seq;

// Operand images kept across calls (pkv_pool_set_image_cache).  A slot
// holds one 64-key tile's images for every kv head; `map` finds the slot of a
// tile key (layer, length, offset in the first page, and each covering page
// with its write generation), `lru` orders the occupied slots, most recently
// used first.
struct ImageCache {
    int32_t n_slots = 0;  // 0: off
    size_t slot_bytes = 0;
    DevBuf buf;
    std::unordered_map<std::string, int32_t> map;
    std::vector<std::string> key_of;
    std::list<int32_t> lru;
    std::vector<std::list<int32_t>::iterator> where;
    std::vector<char> in_lru;
    std::vector<int32_t> free_slots;

    void reset(int32_t n) {
        n_slots = n;
        map.clear();
        lru.clear();
        key_of.assign(n, std::string());
        where.assign(n, lru.end());
        in_lru.assign(n, 0);
        free_slots.clear();
        for (int32_t i = n - 1; i >= 0; --i) free_slots.push_back(i);
    }
    // The slot of `key`; `hit` tells whether it already holds the images.  A
    // miss takes a free slot or the least recently used one.
    int32_t get(const std::string &key, bool &hit) {
        auto it = map.find(key);
        int32_t slot;
        if (it != map.end()) {
            hit = true;
            slot = it->second;
            lru.erase(where[slot]);
        } else {
            hit = false;
            if (!free_slots.empty()) {
                slot = free_slots.back();
                free_slots.pop_back();
            } else {
                slot = lru.back();
                lru.pop_back();
                map.erase(key_of[slot]);
            }
            key_of[slot] = key;
            map.emplace(key, slot);
        }
        lru.push_front(slot);
        where[slot] = lru.begin();
        in_lru[slot] = 1;
        return slot;
    }
};

struct pkv_pool {
    int32_t n_blocks = 0, n_layers = 0, kv_dim = 0, bs = 0, bs_shift = -1;
    int32_t max_seqs = 0, max_blocks = 0;
    bool host_only = false;
    void *k = nullptr, *v = nullptr;
    bool owns_kv = false;
    bool bf16 = false;  // storage element: f32, or bf16 (PKV_POOL_BF16)
    bool fp8 = false;   // or fp8 e4m3 of x / kv_scale (PKV_POOL_FP8)
    float kv_scale = 1.f;
    int32_t *pt_dev = nullptr;
    int32_t *err_dev = nullptr;
    cudaStream_t stream = nullptr;
    int device = 0;
    int n_sm = 0;  // the device's SM count (sizes the shared-prefix pass)

    int64_t last_work[PKV_WORK_FIELDS] = {};  // work list of the last attend call
    std::vector<uint32_t> gen;  // write generation per (block, layer)
    ImageCache icache;

    std::vector<int32_t> free_stack;   // top = back
    std::vector<int32_t> refcnt;
    std::vector<int32_t> free_slots;   // top = back
    std::vector<pkv_seq *> slot_owner;
    std::vector<pkv_seq *> dirty;      // sequences with page-table entries not yet uploaded

    Stager stager;
    DevBuf desc, part, io_in, io_out, qrot, img;
    Blob blob;

    int64_t block_floats() const { return static_cast<int64_t>(n_layers) * bs * kv_dim; }  // elements
    size_t elem_bytes() const { return fp8 ? 1 : bf16 ? 2 : 4; }
    bool narrow() const { return bf16 || fp8; }  // a storage element other than f32
};

struct pkv_seq {
    pkv_pool *pool = nullptr;
    int32_t slot = -1, len = 0, max_tokens = 0;
    std::vector<int32_t> pt;
    int32_t dlo = 0, dhi = 0;
    bool dirty = false;
};

namespace {

void mark_dirty(pkv_seq *s, int32_t lo, int32_t hi) {
    pkv_pool *p = s->pool;
    if (p->host_only || hi <= lo) return;
    if (!s->dirty) {
        s->dirty = true;
        s->dlo = lo;
        s->dhi = hi;
        p->dirty.push_back(s);
    } else {
        s->dlo = std::min(s->dlo, lo);
        s->dhi = std::max(s->dhi, hi);
    }
}

// A page about to receive new contents (a fresh block, a copy-on-append
// target, appended rows): images made from its old contents are stale.
void bump_gen(pkv_pool *p, int32_t b, int32_t layer) {
    if (p->gen.empty()) return;
    if (layer >= 0) {
        ++p->gen[static_cast<size_t>(b) * p->n_layers + layer];
    } else {
        for (int32_t l = 0; l < p->n_layers; ++l) ++p->gen[static_cast<size_t>(b) * p->n_layers + l];
    }
}

int32_t pop_block(pkv_pool *p) {
    if (p->free_stack.empty()) return -1;
    int32_t b = p->free_stack.back();
    p->free_stack.pop_back();
    p->refcnt[b] = 1;
    bump_gen(p, b, -1);
    return b;
}

void unref(pkv_pool *p, int32_t b) {
    if (--p->refcnt[b] == 0) p->free_stack.push_back(b);
}

// Page-table changes since the last upload, as runs into the blob.
void put_pt_runs(pkv_pool *p, Blob &blob, size_t *runs_off, int32_t *n_runs, size_t *vals_off) {
    std::vector<PtRun> runs;
    std::vector<int32_t> vals;
    for (pkv_seq *s : p->dirty) {
        const int32_t hi = std::min<int32_t>(s->dhi, static_cast<int32_t>(s->pt.size()));
        if (hi > s->dlo) {
            runs.push_back({s->slot, s->dlo, hi - s->dlo, static_cast<int32_t>(vals.size())});
            vals.insert(vals.end(), s->pt.begin() + s->dlo, s->pt.begin() + hi);
        }
        s->dirty = false;
    }
    p->dirty.clear();
    *runs_off = blob.put(runs.data(), runs.size());
    *vals_off = blob.put(vals.data(), vals.size());
    *n_runs = static_cast<int32_t>(runs.size());
}

PagedAddr paged_addr(const pkv_pool *p, int32_t layer) {
    PagedAddr a;
    a.k = p->k;
    a.v = p->v;
    a.bf16 = p->bf16 ? 1 : 0;
    a.fp8 = p->fp8 ? 1 : 0;
    a.kv_scale = p->kv_scale;
    a.pt = p->pt_dev;
    a.block_stride = p->block_floats();
    a.layer_off = static_cast<int64_t>(layer) * p->bs * p->kv_dim;
    a.kv_dim = p->kv_dim;
    a.bs = p->bs;
    a.bs_shift = p->bs_shift;
    a.max_blocks = p->max_blocks;
    a.n_blocks = p->n_blocks;
    return a;
}

// Rows [len, len+n) lie in existing blocks of refcount 1.
bool can_append(const pkv_seq *s, int32_t n) {
    const pkv_pool *p = s->pool;
    if (static_cast<int64_t>(s->len) + n > static_cast<int64_t>(s->pt.size()) * p->bs) return false;
    for (int32_t k = s->len / p->bs; k <= (s->len + n - 1) / p->bs; ++k)
        if (p->refcnt[s->pt[k]] != 1) return false;
    return true;
}

// The second tile of a CTA that has only one.
constexpr PrefillTile kNoTile{-1, 0, 0, -1, 0};

int64_t count_tiles(const std::vector<PrefillTile> &v) {
    return std::count_if(v.begin(), v.end(), [](const PrefillTile &t) { return t.row >= 0; });
}

// Work list for a set of rows.  Rows with many queries (and a supported
// shape) become tensor-core prefill tiles; every other query becomes split-K
// decode units, listed longest first; prefill tiles are listed latest-first
// (the latest queries see the most keys), two per tensor-core CTA.
struct WorkList {
    std::vector<UnitDesc> units;
    std::vector<PrefillTile> tiles;
    std::vector<PrefillTile> ctiles;  // shared-prefix pass (non-causal, split S)
    std::vector<MergeDesc> merges;   // queries with several splits (decode first, then prefill)
    std::vector<MergeDesc> pmerges;  // prefill items while building
    int64_t n_part = 0;
};

// A run of consecutive single-query rows whose page tables start with the
// same Lp / bs pages (shared through forks: a page id common to two live
// sequences is one physical page, so those keys are identical).
struct Cascade {
    int32_t r0, n, Lp;
};

// Shared-prefix groups of a decode batch: at least kCascadeMinRows
// consecutive rows with one query each whose first kCascadeMinKeys or more
// keys lie in common whole pages.  The group's common page count is fixed by
// its first two rows; later rows join while they share all of those pages.
constexpr int32_t kCascadeMinRows = 16;
constexpr int32_t kCascadeMinKeys = 2048;

std::vector<Cascade> find_cascades(pkv_seq *const *seqs, int32_t M, const int32_t *n_q,
                                   int32_t bs) {
    std::vector<Cascade> out;
    auto eligible = [&](int32_t r) { return n_q[r] == 1 && seqs[r]->len >= kCascadeMinKeys; };
    auto shares = [&](int32_t a, int32_t b, int32_t pages) {
        const std::vector<int32_t> &x = seqs[a]->pt, &y = seqs[b]->pt;
        return seqs[b]->len / bs >= pages &&
               std::equal(x.begin(), x.begin() + pages, y.begin());
    };
    int32_t r = 0;
    while (r + 1 < M) {
        if (!eligible(r) || !eligible(r + 1)) {
            ++r;
            continue;
        }
        const std::vector<int32_t> &x = seqs[r]->pt, &y = seqs[r + 1]->pt;
        int32_t lim = std::min(seqs[r]->len, seqs[r + 1]->len) / bs;
        int32_t pages = 0;
        while (pages < lim && x[pages] == y[pages]) ++pages;
        if (static_cast<int64_t>(pages) * bs < kCascadeMinKeys) {
            ++r;
            continue;
        }
        int32_t e = r + 2;
        while (e < M && eligible(e) && shares(r, e, pages)) ++e;
        const int32_t n = e - r, Lp = pages * bs;
        if (n >= kCascadeMinRows && Lp >= n) {
            out.push_back({r, n, Lp});
            r = e;
        } else {
            ++r;
        }
    }
    return out;
}

// Keys per split of the shared-prefix pass.  Its CTAs (pair of query tiles x
// kv head x split) each pay a fixed cost -- loading and splitting the query
// rows, writing the partial rows -- worth about kPrefixCtaTiles 64-key tiles
// of work, so the split count of the longest prefix is the one that minimises
// rounds x (tiles per CTA + that cost) on the device's SMs: for 128 forks of
// an 8192-token prefix (16 CTAs per split on 152 SMs), 9 splits of 960 keys
// in one round.
constexpr int32_t kPrefixCtaTiles = 7;
int32_t prefix_split_keys(const std::vector<Cascade> &cas, int32_t group, int32_t n_kv, int32_t n_sm) {
    const int32_t TQ = 128 / group;
    int64_t per_split = 0;  // CTAs per split, all runs
    int32_t lp = 0;
    for (const Cascade &c : cas) {
        per_split += static_cast<int64_t>(ceil_div(ceil_div(c.n, TQ), 2)) * n_kv;  // tile pairs
        lp = std::max(lp, c.Lp);
    }
    const int32_t tiles = ceil_div(lp, kKeyTile);
    const int64_t sms = std::max(1, n_sm);
    int32_t best_ns = 1;
    int64_t best = -1;
    for (int32_t ns = 1; ns <= tiles; ++ns) {
        const int64_t rounds = (ns * per_split + sms - 1) / sms;
        const int64_t cost = rounds * (ceil_div(tiles, ns) + kPrefixCtaTiles);
        if (best < 0 || cost < best) {
            best = cost;
            best_ns = ns;
        }
    }
    return ceil_div(tiles, best_ns) * kKeyTile;
}

// Work of the cascade groups: per group one virtual row (the members' queries,
// consecutive in Q, over keys [0, Lp), non-causal) cut into tensor-core tiles
// of split Sp, and per member the decode units of keys [Lp, total_k) and a
// merge item whose records are the prefix splits followed by the suffix
// splits.  Members get k0 = Lp, s0 = the prefix split count; virtual rows are
// appended to `rows`.  Returns the member mask.
std::vector<char> add_cascades(std::vector<RowDesc> &rows, const std::vector<Cascade> &cas,
                               int32_t S, int32_t Sp, int32_t group, WorkList &w,
                               std::vector<UnitDesc> &tail) {
    std::vector<char> member(rows.size(), 0);
    const int32_t TQ = 128 / group;
    for (const Cascade &c : cas) {
        const int32_t n_pref = ceil_div(c.Lp, Sp);
        int32_t max_suf = 0;
        for (int32_t t = 0; t < c.n; ++t) {
            const RowDesc &rd = rows[c.r0 + t];
            max_suf = std::max(max_suf, ceil_div(rd.past_len + rd.n_q - c.Lp, S));
        }
        const int32_t stride = n_pref + max_suf;
        const int32_t part0 = static_cast<int32_t>(w.n_part);
        w.n_part += static_cast<int64_t>(c.n) * stride;
        RowDesc vr{rows[c.r0].slot, c.Lp - c.n, c.n, rows[c.r0].q_row0};
        const int32_t vi = static_cast<int32_t>(rows.size());
        rows.push_back(vr);
        // split-major: the query tiles that read the same prefix keys (the
        // same operand images) are neighbours in the grid, so they run
        // together and share those images in L2; two neighbouring tiles per
        // CTA (the second absent past the last tile)
        for (int32_t sp = 0; sp < n_pref; ++sp)
            for (int32_t q0 = 0; q0 < c.n; q0 += 2 * TQ) {
                w.ctiles.push_back({vi, q0, sp, part0 + q0 * stride, stride});
                const int32_t q1 = q0 + TQ;
                w.ctiles.push_back(q1 < c.n ? PrefillTile{vi, q1, sp, part0 + q1 * stride, stride} : kNoTile);
            }
        for (int32_t t = 0; t < c.n; ++t) {
            const int32_t r = c.r0 + t;
            RowDesc &rd = rows[r];
            const int32_t n_suf = ceil_div(rd.past_len + rd.n_q - c.Lp, S);
            rd.k0 = c.Lp;
            rd.s0 = n_pref;
            const int32_t item = static_cast<int32_t>(w.merges.size());
            w.merges.push_back({r, 0, part0 + t * stride, n_pref + n_suf});
            for (int32_t j = 0; j + 1 < n_suf; ++j) w.units.push_back({r, 0, n_pref + j, item});
            tail.push_back({r, 0, n_pref + n_suf - 1, item});
            member[r] = 1;
        }
    }
    return member;
}

// Keys of one decode unit (the host's copy of the kernels' unit_range).
int32_t unit_keys(const UnitDesc &u, const RowDesc &rd, int causal, int32_t S) {
    const int32_t total_k = rd.past_len + rd.n_q;
    const int32_t lim = causal ? total_k - rd.n_q + u.qi + 1 : total_k;
    const int32_t kbeg = rd.k0 + (u.split - rd.s0) * S;
    return std::max(0, std::min(kbeg + S, lim) - kbeg);
}

// Cost of a tensor-core prefill CTA in units of ~100 SM clocks, from clock64
// timelines of the kernel: ~3.9k clocks per 64-key tile with two chains,
// ~2.7k with one, ~15k per CTA besides (query rows, first copies, output).
constexpr int64_t kPairTileCost = 39, kSingleTileCost = 27, kCtaCost = 150;

// Tile pairs -> the CTA list (two entries per CTA, the second may be absent).
// mode 0: one tile per CTA; 1: every pair; 2: pairs, with the last k of the
// list split into two one-tile CTAs (which then run last, beside the pairs
// that read the same rows' images, so those are still in L2) where that ends
// the launch sooner on n_sm SMs (the hardware hands CTAs to free SMs in
// order; every entry is n_kv CTAs).
// A chain's arithmetic does not depend on its partner, so the outputs are the
// same bits in every mode.
void place_pairs(const std::vector<std::array<PrefillTile, 2>> &pairs, const std::vector<int32_t> &len0,
                 const std::vector<int32_t> &len1, int32_t mode, int32_t n_kv, int32_t n_sm,
                 std::vector<PrefillTile> &out) {
    const size_t np = pairs.size();
    if (mode == 0) {
        for (const auto &pr : pairs)
            for (const PrefillTile &t : pr)
                if (t.row >= 0) {
                    out.push_back(t);
                    out.push_back(kNoTile);
                }
        return;
    }
    std::vector<size_t> full;  // pairs with both tiles, last in the list first
    for (size_t i = np; i-- > 0;)
        if (pairs[i][1].row >= 0) full.push_back(i);
    const int64_t ctas = static_cast<int64_t>(np) * std::max(1, n_kv);
    const int64_t rounds = n_sm > 0 ? (ctas + n_sm - 1) / n_sm : 0;
    int32_t best_k = 0;
    if (mode == 2 && n_sm > 0 && n_kv > 0 && !full.empty() && rounds <= 16) {
        std::vector<char> split(np, 0);
        std::vector<int64_t> heap;
        // finish time of the launch with the last k pairs split: pairs (and
        // one-tile entries) in list order, then the split tiles in list order
        auto makespan = [&](int32_t k) {
            std::fill(split.begin(), split.end(), 0);
            for (int32_t i = 0; i < k; ++i) split[full[i]] = 1;
            heap.assign(static_cast<size_t>(n_sm), 0);
            auto put = [&](int64_t cost) {
                for (int32_t h = 0; h < n_kv; ++h) {
                    std::pop_heap(heap.begin(), heap.end(), std::greater<int64_t>());
                    heap.back() += cost;
                    std::push_heap(heap.begin(), heap.end(), std::greater<int64_t>());
                }
            };
            for (size_t i = 0; i < np; ++i) {
                if (split[i]) continue;
                const bool two = pairs[i][1].row >= 0;
                put(two ? kPairTileCost * std::max(len0[i], len1[i]) + kCtaCost
                        : kSingleTileCost * len0[i] + kCtaCost);
            }
            for (int32_t i = k - 1; i >= 0; --i) {
                put(kSingleTileCost * len0[full[i]] + kCtaCost);
                put(kSingleTileCost * len1[full[i]] + kCtaCost);
            }
            return *std::max_element(heap.begin(), heap.end());
        };
        int64_t best = makespan(0);
        for (int64_t r = 1; r <= rounds; ++r) {
            const int64_t keep = r * n_sm / n_kv;  // pair entries that fill r rounds
            const int32_t k = static_cast<int32_t>(std::max<int64_t>(0, std::min<int64_t>(
                static_cast<int64_t>(full.size()), static_cast<int64_t>(np) - keep)));
            if (k == 0) continue;
            const int64_t t = makespan(k);
            if (t < best) {
                best = t;
                best_k = k;
            }
        }
    }
    std::vector<char> split(np, 0);
    for (int32_t i = 0; i < best_k; ++i) split[full[i]] = 1;
    for (size_t i = 0; i < np; ++i)
        if (!split[i]) {
            out.push_back(pairs[i][0]);
            out.push_back(pairs[i][1]);
        }
    for (int32_t i = best_k - 1; i >= 0; --i)
        for (const PrefillTile &t : pairs[full[i]]) {
            out.push_back(t);
            out.push_back(kNoTile);
        }
}

// S: keys per split-K decode unit; prefill_split: keys per split of the
// tensor-core prefill rows (0: kPrefillSplitFactor * S); prefix_split: keys
// per split of the shared-prefix pass (0: S); allow_tc false: every row to the
// split-K decode kernels; n_kv, n_sm: kv heads and the device's SMs, for the
// placement of the prefill tiles (0: not known).
void build_work(std::vector<RowDesc> &rows, int causal, int32_t S, int32_t head_dim,
                int32_t group, WorkList &w, const std::vector<Cascade> &cas = {},
                int32_t prefix_split = 0, int32_t prefill_split = 0, bool allow_tc = true,
                int32_t n_kv = 0, int32_t n_sm = 0) {
    std::vector<UnitDesc> tail;
    w.units.clear();
    w.tiles.clear();
    w.ctiles.clear();
    w.merges.clear();
    w.pmerges.clear();
    w.n_part = 0;
    const int32_t n_real = static_cast<int32_t>(rows.size());
    const std::vector<char> member =
        add_cascades(rows, cas, S, prefix_split > 0 ? prefix_split : S, group, w, tail);
    const bool tc_shape = allow_tc && prefill_shape(head_dim, group);
    const int32_t TQ = tc_shape ? 128 / group : 0;
    const int32_t Sp = prefill_split > 0 ? prefill_split : S * kPrefillSplitFactor;
    std::vector<std::array<PrefillTile, 2>> pairs;
    std::vector<int32_t> len0, len1;  // key tiles of each pair's tiles
    auto key_tiles = [&](const PrefillTile &t) {
        if (t.row < 0) return 0;
        const RowDesc &rd = rows[t.row];
        const int32_t total_k = rd.past_len + rd.n_q, nv = std::min(TQ, rd.n_q - t.q0);
        const int32_t kend_tile = causal ? std::min(total_k, total_k - rd.n_q + t.q0 + nv) : total_k;
        const int32_t kbeg = t.split * Sp, kend = std::min(kbeg + Sp, kend_tile);
        return std::max(0, ceil_div(kend, kKeyTile) - kbeg / kKeyTile);
    };
    for (int32_t r = 0; r < n_real; ++r) {
        if (member[r]) continue;
        const RowDesc &rd = rows[r];
        const int32_t total_k = rd.past_len + rd.n_q;
        if (tc_shape && rd.n_q >= kPrefillMinQueries) {
            // query tiles latest first (part0 -1: one split, written directly)
            struct QTile {
                int32_t q0, ns, part0;
            };
            std::vector<QTile> qt;
            for (int32_t q0 = ((rd.n_q - 1) / TQ) * TQ; q0 >= 0; q0 -= TQ) {
                const int32_t nv = std::min(TQ, rd.n_q - q0);
                const int32_t kend = causal ? total_k - rd.n_q + q0 + nv : total_k;
                const int32_t ns = ceil_div(kend, Sp);
                int32_t part0 = -1;
                if (ns > 1) {
                    part0 = static_cast<int32_t>(w.n_part);
                    w.n_part += static_cast<int64_t>(nv) * ns;
                    for (int32_t t = 0; t < nv; ++t) w.pmerges.push_back({r, q0 + t, part0 + t * ns, ns});
                }
                qt.push_back({q0, ns, part0});
            }
            // neighbouring tiles in pairs, one CTA per pair and split (the
            // pair's tiles of one split share every key tile); a present tile
            // first, the second absent where a tile has no partner
            for (size_t i = 0; i < qt.size(); i += 2) {
                const QTile &x = qt[i];
                const QTile *y = i + 1 < qt.size() ? &qt[i + 1] : nullptr;
                const int32_t ns = std::max(x.ns, y ? y->ns : 0);
                for (int32_t sp = 0; sp < ns; ++sp) {
                    PrefillTile u = sp < x.ns ? PrefillTile{r, x.q0, sp, x.part0} : kNoTile;
                    PrefillTile v = y && sp < y->ns ? PrefillTile{r, y->q0, sp, y->part0} : kNoTile;
                    if (u.row < 0) std::swap(u, v);
                    pairs.push_back({u, v});
                    len0.push_back(key_tiles(u));
                    len1.push_back(key_tiles(v));
                }
            }
            continue;
        }
        for (int32_t i = 0; i < rd.n_q; ++i) {
            const int32_t q_pos = total_k - rd.n_q + i;
            const int32_t nk = causal ? q_pos + 1 : total_k;
            const int32_t ns = ceil_div(nk, S);
            if (ns == 1) {
                tail.push_back({r, i, 0, -1});
            } else {
                const int32_t part0 = static_cast<int32_t>(w.n_part);
                const int32_t item = static_cast<int32_t>(w.merges.size());
                w.n_part += ns;
                w.merges.push_back({r, i, part0, ns});
                for (int32_t s = 0; s + 1 < ns; ++s) w.units.push_back({r, i, s, item});
                tail.push_back({r, i, ns - 1, item});
            }
        }
    }
    place_pairs(pairs, len0, len1, g_prefill_pairing.load(), n_kv, n_sm, w.tiles);
    w.units.insert(w.units.end(), tail.begin(), tail.end());
    // longest units first, so that the grid's last CTAs are its shortest and
    // the launch drains quickly (the order changes no result)
    {
        std::vector<std::pair<int32_t, int32_t>> key(w.units.size());
        for (size_t i = 0; i < w.units.size(); ++i)
            key[i] = {-unit_keys(w.units[i], rows[w.units[i].row], causal, S), static_cast<int32_t>(i)};
        std::sort(key.begin(), key.end());
        std::vector<UnitDesc> sorted(w.units.size());
        for (size_t i = 0; i < key.size(); ++i) sorted[i] = w.units[key[i].second];
        w.units.swap(sorted);
    }
    // one merge list: decode items first (units refer to them by index), then prefill items
    w.merges.insert(w.merges.end(), w.pmerges.begin(), w.pmerges.end());
    w.pmerges.clear();
}

// The fused append may replace the page-table upload when every pending
// change belongs to a sequence of this batch and lies in pages that hold none
// of its past positions and only positions this call appends: nothing in the
// launch reads those entries (new positions come from K_new / V_new), and the
// kernel enters them itself.
bool dirty_within_appends(const pkv_pool *p, pkv_seq *const *seqs, int32_t M, const int32_t *n_q) {
    std::unordered_map<const pkv_seq *, int32_t> row_of;
    for (int32_t r = 0; r < M; ++r) row_of[seqs[r]] = r;
    for (const pkv_seq *s : p->dirty) {
        const auto it = row_of.find(s);
        if (it == row_of.end()) return false;
        const int32_t hi = std::min<int32_t>(s->dhi, static_cast<int32_t>(s->pt.size()));
        if (hi <= s->dlo) continue;
        const int32_t first_new = ceil_div(s->len, p->bs);
        const int32_t end_new = ceil_div(s->len + n_q[it->second], p->bs);
        if (s->dlo < first_new || hi > end_new) return false;
    }
    return true;
}

// Mark every pending page-table change as uploaded; true if there was one.
bool clear_dirty(pkv_pool *p) {
    bool any = false;
    for (pkv_seq *s : p->dirty) {
        any = any || s->dhi > s->dlo;
        s->dirty = false;
    }
    p->dirty.clear();
    return any;
}

int check_heads(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim) {
    if (n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return fail(PKV_ERR_BAD_DIM, "n_heads, n_kv_heads and head_dim must be positive");
    if (n_heads % n_kv_heads != 0)
        return fail(PKV_ERR_BAD_GQA, "n_heads (%d) is not a multiple of n_kv_heads (%d)", n_heads,
                    n_kv_heads);
    return PKV_OK;
}

int check_dup(const pkv_pool *p, pkv_seq *const *seqs, int32_t M) {
    std::vector<char> seen(p->max_seqs, 0);
    for (int32_t r = 0; r < M; ++r) {
        if (seen[seqs[r]->slot]) return fail(PKV_ERR_ARG, "sequence appears twice in the batch");
        seen[seqs[r]->slot] = 1;
    }
    return PKV_OK;
}

// Upload the blob to the pool's descriptor buffer.
cudaError_t upload_blob(pkv_pool *p) {
    cudaError_t e = p->desc.ensure(p->blob.size(), p->stream, p->device);
    if (e != cudaSuccess) return e;
    return p->stager.upload(p->desc.p, p->blob.b.data(), p->blob.b.size(), p->stream);
}

template <class T>
const T *dptr(const pkv_pool *p, size_t off) {
    return reinterpret_cast<const T *>(static_cast<unsigned char *>(p->desc.p) + off);
}

// Argument checks of a layer call, before it changes anything, in the order
// of nx_f32_attn_with_paged: sizes, grouping, sequence.
int validate_layer(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q,
                   const float *K_new, const float *V_new, int32_t n_heads, int32_t n_kv_heads,
                   int32_t head_dim, int32_t layer, const float *out, bool host_io, bool attend,
                   double rope_base) {
    if (M <= 0 || !n_q) return fail(PKV_ERR_BAD_DIM, "M must be positive and n_q non-NULL");
    for (int32_t r = 0; r < M; ++r)
        if (n_q[r] <= 0) return fail(PKV_ERR_BAD_DIM, "n_q[%d] = %d must be positive", r, n_q[r]);
    if (attend) {
        int rc = check_heads(n_heads, n_kv_heads, head_dim);
        if (rc) return rc;
        if (rope_base < 0.0 || (rope_base > 0.0 && (head_dim % 2) != 0))
            return fail(rope_base < 0.0 ? PKV_ERR_ARG : PKV_ERR_BAD_DIM,
                        "RoPE needs a positive base and an even head_dim");
    }
    if (!seqs) return fail(PKV_ERR_SEQ, "seqs is NULL");
    for (int32_t r = 0; r < M; ++r)
        if (!seqs[r] || !seqs[r]->pool) return fail(PKV_ERR_SEQ, "sequence %d is NULL", r);
    pkv_pool *p = seqs[0]->pool;
    for (int32_t r = 1; r < M; ++r)
        if (seqs[r]->pool != p) return fail(PKV_ERR_ARG, "sequences of different pools in one batch");
    if (p->host_only) return fail(PKV_ERR_ARG, "host-only pool has no device storage");
    if (attend) {
        if (static_cast<int64_t>(n_kv_heads) * head_dim != p->kv_dim)
            return fail(PKV_ERR_BAD_DIM, "n_kv_heads*head_dim = %d differs from the pool's kv_dim %d",
                        n_kv_heads * head_dim, p->kv_dim);
        if (head_dim > kMaxHeadDim)
            return fail(PKV_ERR_BAD_DIM, "head_dim %d > %d is not supported", head_dim, kMaxHeadDim);
        if (p->fp8 && head_dim == 128 && (p->kv_dim % 16) != 0)
            return fail(PKV_ERR_BAD_DIM, "an fp8 pool with head_dim 128 needs kv_dim %% 16 == 0");
    }
    if (layer < 0 || layer >= p->n_layers)
        return fail(PKV_ERR_ARG, "layer %d outside [0, %d)", layer, p->n_layers);
    if (!K_new || !V_new || (attend && (!Q || !out)))
        return fail(PKV_ERR_ARG, "NULL data pointer");
    if (!host_io) {
        // 16-byte alignment where the kernels use vector access (head_dim % 4 == 0),
        // element alignment otherwise
        const bool vec = attend && (head_dim % 4) == 0;
        auto ok = [&](const void *q) { return vec ? aligned16(q) : aligned4(q); };
        if (!ok(K_new) || !ok(V_new) || (attend && (!ok(Q) || !ok(out))))
            return fail(PKV_ERR_ARG, vec ? "device pointers must be 16-byte aligned"
                                         : "device pointers must be 4-byte aligned");
    }
    {
        int rc = check_dup(p, seqs, M);
        if (rc) return rc;
    }
    for (int32_t r = 0; r < M; ++r)
        if (!can_append(seqs[r], n_q[r]))
            return fail(PKV_ERR_SEQ, "rows [%d, %d) of batch row %d are not ensured (call pkv_ensure_append)",
                        seqs[r]->len, seqs[r]->len + n_q[r], r);
    return PKV_OK;
}

// Shared body of pkv_attn_batch / pkv_attn_with_paged / pkv_attn_batch_host /
// pkv_append_layer.  `attend` = false stops after the append.
int run_layer(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q,
              const float *K_new, const float *V_new, int32_t n_heads, int32_t n_kv_heads,
              int32_t head_dim, int32_t layer, int32_t causal, float scale, float *out,
              bool host_io, bool attend, double rope_base = 0.0) {
    {
        const int rc = validate_layer(seqs, M, n_q, Q, K_new, V_new, n_heads, n_kv_heads, head_dim,
                                      layer, out, host_io, attend, rope_base);
        if (rc) return rc;
    }
    pkv_pool *p = seqs[0]->pool;
    DevGuard dg(p->device);
    cudaStream_t st = p->stream;
    const int32_t q_dim = n_heads * head_dim;
    const int32_t kv_dim = p->kv_dim;

    std::vector<RowDesc> rows(M);
    std::vector<AppendDesc> app;
    int64_t T = 0;
    for (int32_t r = 0; r < M; ++r) {
        rows[r] = {seqs[r]->slot, seqs[r]->len, n_q[r], static_cast<int32_t>(T)};
        for (int32_t t = 0; t < n_q[r]; ++t) {
            const int32_t pos = seqs[r]->len + t;
            app.push_back({seqs[r]->slot, pos, static_cast<int32_t>(T + t), seqs[r]->pt[pos / p->bs]});
        }
        T += n_q[r];
    }
    if (T > 0x7fffffffLL / std::max(q_dim, kv_dim)) return fail(PKV_ERR_BAD_DIM, "batch too large");

    WorkList w;
    const int32_t S = g_split_keys.load();
    // A decode unit covers the same bytes of K/V on every pool: S keys of f32
    // rows, 2 S of bf16, 4 S of fp8 (so a unit's fixed work -- the query
    // pieces, the 4-warp merge -- is amortised alike).  It depends on the
    // pool only, so a row's split boundaries are the same in any batch.
    const int32_t S_dec = std::min<int32_t>(65536, S * (p->fp8 ? 4 : p->bf16 ? 2 : 1));
    const int32_t group = attend ? n_heads / n_kv_heads : 0;
    std::vector<Cascade> cas;
    if (attend && g_cascade.load() != 0 && prefill_shape(head_dim, group))
        cas = find_cascades(seqs, M, n_q, p->bs);
    const int32_t Sp = cas.empty() ? 0 : prefix_split_keys(cas, group, n_kv_heads, p->n_sm);
    if (attend)
        build_work(rows, causal, S_dec, head_dim, group, w, cas, Sp, S * kPrefillSplitFactor, true, n_kv_heads,
                   p->n_sm);
    // the decode kernels that take the append themselves: the f32 kernel for
    // groups 1, 2, 4 and the narrow-pool kernel for its shapes (head_dim 128)
    const bool fuse_shape = head_dim == 128 &&
                            (p->narrow() ? decode_mma_shape(head_dim, group, p->bf16, p->fp8)
                                         : (group == 1 || group == 2 || group == 4));
    const bool fuse = attend && rope_base == 0.0 && g_fused_append.load() != 0 && w.tiles.empty() &&
                      w.ctiles.empty() && !w.units.empty() && fuse_shape &&
                      dirty_within_appends(p, seqs, M, n_q);

    if (attend) {
        int64_t pairs = 0, ppairs = 0;
        for (int32_t r = 0; r < M; ++r) {
            const RowDesc &rd = rows[r];
            if (rd.n_q < kPrefillMinQueries || !prefill_shape(head_dim, group)) continue;
            const int64_t n = rd.n_q, b = rd.past_len;
            pairs += causal ? n * b + n * (n + 1) / 2 : n * (b + n);
        }
        for (const Cascade &c : cas) ppairs += static_cast<int64_t>(c.n) * c.Lp;
        const int64_t vals[PKV_WORK_FIELDS] = {static_cast<int64_t>(w.units.size()),
                                               count_tiles(w.tiles),
                                               count_tiles(w.ctiles),
                                               static_cast<int64_t>(w.merges.size()),
                                               pairs, ppairs, fuse ? 1 : 0, 0, 0, Sp,
                                               static_cast<int64_t>(w.tiles.size() / 2) * n_kv_heads};
        std::copy(vals, vals + PKV_WORK_FIELDS, p->last_work);
    }

    // the pages this call writes get new generations
    for (const AppendDesc &ad : app) bump_gen(p, ad.blk, layer);

    // operand images for the tensor-core launches: every 64-key tile of each
    // row with prefill tiles (real rows and shared-prefix virtual rows).  Tile
    // kt of row r is image img_slot[img_tile0[r] + kt]; the split pass builds
    // the ones listed in split_items.  With the image cache, a tile whose
    // pages are unchanged since an earlier call keeps that call's image.
    std::vector<int32_t> img_tile0, img_slot;
    std::vector<SplitItem> split_items;
    bool cached = false;
    int64_t img_hits = 0;
    if (!w.tiles.empty() || !w.ctiles.empty()) {
        img_tile0.assign(rows.size(), -1);
        std::vector<int32_t> order;  // rows needing images, first use first
        int32_t next = 0;
        auto need = [&](int32_t r) {
            if (img_tile0[r] >= 0) return;
            img_tile0[r] = next;
            next += ceil_div(rows[r].past_len + rows[r].n_q, kKeyTile);
            order.push_back(r);
        };
        for (const PrefillTile &t : w.tiles)
            if (t.row >= 0) need(t.row);
        for (const PrefillTile &t : w.ctiles)
            if (t.row >= 0) need(t.row);
        img_slot.resize(next);
        ImageCache &ic = p->icache;
        cached = ic.n_slots >= next && ic.slot_bytes == static_cast<size_t>(n_kv_heads) * kImageBytes;
        // the host page table of each row: a shared-prefix virtual row reads
        // its first member's (add_cascades appends them in cascade order)
        auto row_seq = [&](int32_t r) { return r < M ? seqs[r] : seqs[cas[r - M].r0]; };
        std::string key;
        for (int32_t r : order) {
            const int32_t tk = rows[r].past_len + rows[r].n_q, nt = ceil_div(tk, kKeyTile);
            const pkv_seq *sq = row_seq(r);
            for (int32_t kt = 0; kt < nt; ++kt) {
                const int32_t i = img_tile0[r] + kt;
                if (!cached) {
                    img_slot[i] = i;
                    split_items.push_back({r, kt, i});
                    continue;
                }
                const int32_t k0 = kt * kKeyTile, nv = std::min(kKeyTile, tk - k0);
                const int32_t g0 = k0 / p->bs, g1 = (k0 + nv - 1) / p->bs;
                key.clear();
                auto put = [&](int32_t v) { key.append(reinterpret_cast<const char *>(&v), sizeof v); };
                put(layer);
                put(nv);
                put(k0 % p->bs);
                for (int32_t g = g0; g <= g1; ++g) {
                    const int32_t b = sq->pt[g];
                    put(b);
                    put(static_cast<int32_t>(p->gen[static_cast<size_t>(b) * p->n_layers + layer]));
                }
                bool hit = false;
                img_slot[i] = ic.get(key, hit);
                if (hit) ++img_hits;
                else split_items.push_back({r, kt, img_slot[i]});
            }
        }
    }
    if (attend) {
        p->last_work[7] = img_hits;
        p->last_work[8] = static_cast<int64_t>(split_items.size());
    }

    Blob &blob = p->blob;
    blob.clear();
    size_t runs_off = 0, vals_off = 0;
    int32_t n_runs = 0;
    bool pt_write = false;
    if (fuse) pt_write = clear_dirty(p);
    else put_pt_runs(p, blob, &runs_off, &n_runs, &vals_off);
    const size_t rows_off = blob.put(rows.data(), rows.size());
    const size_t app_off = blob.put(app.data(), app.size());
    const size_t units_off = blob.put(w.units.data(), w.units.size());
    const size_t tiles_off = blob.put(w.tiles.data(), w.tiles.size());
    const size_t ctiles_off = blob.put(w.ctiles.data(), w.ctiles.size());
    const size_t merges_off = blob.put(w.merges.data(), w.merges.size());
    const size_t tile0_off = blob.put(img_tile0.data(), img_tile0.size());
    const size_t slot_off = blob.put(img_slot.data(), img_slot.size());
    const size_t split_off = blob.put(split_items.data(), split_items.size());

    cudaError_t e = upload_blob(p);
    if (e != cudaSuccess) return cuda_fail(e, "descriptor upload");

    const float *Qd = Q, *Kd = K_new, *Vd = V_new;
    float *Od = out;
    if (host_io) {
        const size_t in_bytes = static_cast<size_t>(T) * (q_dim + 2 * kv_dim) * sizeof(float);
        e = p->io_in.ensure(in_bytes, st, p->device);
        if (e == cudaSuccess) e = p->io_out.ensure(static_cast<size_t>(T) * q_dim * sizeof(float), st, p->device);
        if (e != cudaSuccess) return cuda_fail(e, "staging buffers");
        float *base = static_cast<float *>(p->io_in.p);
        float *qd = base, *kd = base + T * q_dim, *vd = kd + T * kv_dim;
        e = cudaMemcpyAsync(qd, Q, sizeof(float) * T * q_dim, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(kd, K_new, sizeof(float) * T * kv_dim, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(vd, V_new, sizeof(float) * T * kv_dim, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "input copy");
        Qd = qd;
        Kd = kd;
        Vd = vd;
        Od = static_cast<float *>(p->io_out.p);
    }

    const PagedAddr addr = paged_addr(p, layer);
    PrepArgs pr{};
    pr.pt = p->pt_dev;
    pr.max_blocks = p->max_blocks;
    pr.runs = dptr<PtRun>(p, runs_off);
    pr.vals = dptr<int32_t>(p, vals_off);
    pr.n_runs = n_runs;
    pr.app = dptr<AppendDesc>(p, app_off);
    pr.n_app = static_cast<int32_t>(T);
    pr.K_new = Kd;
    pr.V_new = Vd;
    pr.vec4 = (kv_dim % 4) == 0 && aligned16(Kd) && aligned16(Vd);
    pr.err = p->err_dev;
    if (attend && rope_base > 0.0) {
        e = p->qrot.ensure(static_cast<size_t>(T) * q_dim * sizeof(float), st, p->device);
        if (e != cudaSuccess) return cuda_fail(e, "rotated-query buffer");
        pr.rope_base = rope_base;
        pr.Q = Qd;
        pr.Q_rot = static_cast<float *>(p->qrot.p);
        pr.q_dim = q_dim;
        pr.hd = head_dim;
        Qd = pr.Q_rot;  // the attention kernels read the rotated queries
    }
    if (!fuse) {
        e = launch(PKV_KERNEL_APPEND, st, [&] { return launch_prep(pr, addr, st); });
        if (e != cudaSuccess) return cuda_fail(e, "prep kernel");
    }
    if (!attend) return PKV_OK;

    AttnArgs a{};
    a.Q = Qd;
    a.out = Od;
    a.rows = dptr<RowDesc>(p, rows_off);
    a.units = dptr<UnitDesc>(p, units_off);
    a.merges = dptr<MergeDesc>(p, merges_off);
    a.n_units = static_cast<int32_t>(w.units.size());
    a.n_heads = n_heads;
    a.n_kv = n_kv_heads;
    a.hd = head_dim;
    a.group = n_heads / n_kv_heads;
    a.causal = causal ? 1 : 0;
    a.split_keys = S_dec;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.err = p->err_dev;
    if (fuse) {
        a.K_new = Kd;
        a.V_new = Vd;
        a.app = pr.app;
        a.pt_write = pt_write ? 1 : 0;
    }
    if (w.n_part > 0) {
        const size_t pf = static_cast<size_t>(w.n_part) * n_heads;
        e = p->part.ensure(pf * (2 + head_dim) * sizeof(float), st, p->device);
        if (e != cudaSuccess) return cuda_fail(e, "partials buffer");
        a.pm = static_cast<float *>(p->part.p);
        a.pl = a.pm + pf;
        a.pacc = a.pl + pf;
    }
    unsigned char *img = nullptr;
    if (!img_slot.empty()) {
        if (cached) {
            img = static_cast<unsigned char *>(p->icache.buf.p);
        } else {
            e = p->img.ensure(img_slot.size() * n_kv_heads * kImageBytes, st, p->device);
            if (e != cudaSuccess) return cuda_fail(e, "operand image buffer");
            img = static_cast<unsigned char *>(p->img.p);
        }
    }
    if (!split_items.empty()) {
        const SplitArgs sa{a.rows, dptr<SplitItem>(p, split_off), static_cast<int32_t>(split_items.size()),
                           n_kv_heads, img, p->err_dev};
        e = launch(PKV_KERNEL_SPLIT, st, [&] { return launch_split_paged(sa, addr, st); });
        if (e != cudaSuccess) {
            if (cached) p->icache.reset(p->icache.n_slots);  // the missed images were not made
            return cuda_fail(e, "split kernel");
        }
    }
    if (!w.tiles.empty()) {
        PrefillArgs pa{Qd, Od, a.rows, dptr<PrefillTile>(p, tiles_off),
                       static_cast<int32_t>(w.tiles.size()), a.pm, a.pl, a.pacc, n_heads,
                       n_kv_heads, a.group, a.causal, S * kPrefillSplitFactor, a.scale_log2,
                       p->err_dev};
        pa.img = img;
        pa.img_tile0 = dptr<int32_t>(p, tile0_off);
        pa.img_slot = dptr<int32_t>(p, slot_off);
        pa.lo_zero = p->narrow() ? 1 : 0;
        e = launch(PKV_KERNEL_PREFILL, st, [&] { return launch_prefill_paged(pa, addr, st); });
        if (e != cudaSuccess) return cuda_fail(e, "prefill kernel");
    }
    if (!w.ctiles.empty()) {
        // shared prefixes: every member query sees all Lp prefix keys
        PrefillArgs pa{Qd, Od, a.rows, dptr<PrefillTile>(p, ctiles_off),
                       static_cast<int32_t>(w.ctiles.size()), a.pm, a.pl, a.pacc, n_heads,
                       n_kv_heads, a.group, 0, Sp, a.scale_log2, p->err_dev};
        pa.img = img;
        pa.img_tile0 = dptr<int32_t>(p, tile0_off);
        pa.img_slot = dptr<int32_t>(p, slot_off);
        pa.lo_zero = p->narrow() ? 1 : 0;
        e = launch(PKV_KERNEL_PREFILL, st, [&] { return launch_prefill_paged(pa, addr, st); });
        if (e != cudaSuccess) return cuda_fail(e, "shared-prefix kernel");
    }
    if (!w.units.empty()) {
        e = launch(PKV_KERNEL_DECODE, st, [&] { return launch_decode_paged(a, addr, st); });
        if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
    }
    if (!w.merges.empty()) {
        MergeArgs m{a.pm, a.pl, a.pacc, Od, a.rows, dptr<MergeDesc>(p, merges_off),
                    static_cast<int32_t>(w.merges.size()), n_heads, head_dim};
        e = launch(PKV_KERNEL_MERGE, st, [&] { return launch_merge(m, st); });
        if (e != cudaSuccess) return cuda_fail(e, "merge kernel");
    }
    if (host_io) {
        e = cudaMemcpyAsync(out, Od, sizeof(float) * T * q_dim, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "output copy");
    }
    return PKV_OK;
}

// The device address of host memory the kernels may read and write directly
// (page-locked memory under unified addressing), or nullptr.
void *device_view(const void *h) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// Host buffers.  Page-locked host memory the device can address is read and
// written by the kernels in place, so those transfers overlap the attention
// work instead of preceding or following it -- where that pays (measured):
//   calls with tensor-core prefill rows: staged copies of everything before
//     and after the launches (a prefill CTA reads 64 KiB of queries before
//     its first MMA and writes 64 KiB of output at its end; over the host
//     link that stalls whole waves, costing more than the copies);
//   decode calls with shared-prefix runs: out written in place (the merge
//     kernel writes it), Q staged (the prefix pass reads it like a prefill);
//   other decode calls: Q read and out written in place;
//   K_new, V_new: always staged (the append reads them once).
// Other host memory takes staged copies before and after the launches.
int run_layer_host(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Qh,
                   const float *Kh, const float *Vh, int32_t n_heads, int32_t n_kv_heads,
                   int32_t head_dim, int32_t layer, int32_t causal, float scale, float *outh) {
    int rc = validate_layer(seqs, M, n_q, Qh, Kh, Vh, n_heads, n_kv_heads, head_dim, layer, outh,
                            true, true, 0.0);
    if (rc) return rc;
    pkv_pool *p = seqs[0]->pool;
    DevGuard dg(p->device);
    const bool vec = (head_dim % 4) == 0;
    auto usable = [&](const void *q) { return q && (vec ? aligned16(q) : aligned4(q)); };
    const int32_t group = n_heads / n_kv_heads;
    bool prefill = false, cascade = false;
    if (prefill_shape(head_dim, group)) {
        for (int32_t r = 0; r < M && !prefill; ++r) prefill = n_q[r] >= kPrefillMinQueries;
        if (!prefill && g_cascade.load() != 0) cascade = !find_cascades(seqs, M, n_q, p->bs).empty();
    }
    float *Ov = prefill ? nullptr : static_cast<float *>(device_view(outh));
    if (!usable(Ov))
        return run_layer(seqs, M, n_q, Qh, Kh, Vh, n_heads, n_kv_heads, head_dim, layer, causal, scale,
                         outh, true, true);
    const float *Qv = cascade ? nullptr : static_cast<const float *>(device_view(Qh));
    if (!usable(Qv)) Qv = nullptr;
    int64_t T = 0;
    for (int32_t r = 0; r < M; ++r) T += n_q[r];
    const int32_t kv_dim = p->kv_dim, q_dim = n_heads * head_dim;
    cudaStream_t st = p->stream;
    const size_t in_floats = static_cast<size_t>(T) * (2 * kv_dim + (Qv ? 0 : q_dim));
    cudaError_t e = p->io_in.ensure(in_floats * sizeof(float), st, p->device);
    if (e != cudaSuccess) return cuda_fail(e, "staging buffers");
    float *kd = static_cast<float *>(p->io_in.p), *vd = kd + T * kv_dim, *qd = vd + T * kv_dim;
    e = cudaMemcpyAsync(kd, Kh, sizeof(float) * T * kv_dim, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(vd, Vh, sizeof(float) * T * kv_dim, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !Qv)
        e = cudaMemcpyAsync(qd, Qh, sizeof(float) * T * q_dim, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "input copy");
    rc = run_layer(seqs, M, n_q, Qv ? Qv : qd, kd, vd, n_heads, n_kv_heads, head_dim, layer, causal,
                   scale, Ov, false, true);
    if (rc != PKV_OK) return rc;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "host-buffer call");
    return PKV_OK;
}

// Contiguous-path globals: one staging ring and error word per device.
std::mutex g_contig_mu;
Stager g_contig_stager[64];
int32_t *g_contig_err[64] = {};

// The error word of pkv_attn_contiguous on device `dev` (current), made and
// cleared on first use.  Call with g_contig_mu held.
cudaError_t contig_error_word(int dev, int32_t **out) {
    if (!g_contig_err[dev]) {
        int32_t *w = nullptr;
        cudaError_t e = cudaMalloc(&w, sizeof(int32_t));
        if (e == cudaSuccess) e = cudaMemset(w, 0, sizeof(int32_t));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            if (w) cudaFree(w);
            return e;
        }
        g_contig_err[dev] = w;
    }
    *out = g_contig_err[dev];
    return cudaSuccess;
}

// Read and clear a device error word (nothing to read when it does not exist
// yet).  The caller has waited for the work that may set it.
cudaError_t take_error_word(int32_t *word, uint32_t *bits) {
    *bits = 0;
    if (!word) return cudaSuccess;
    int32_t h = 0;
    cudaError_t e = cudaMemcpy(&h, word, sizeof h, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && h) e = cudaMemset(word, 0, sizeof h);
    if (e == cudaSuccess && h) e = cudaDeviceSynchronize();
    *bits = static_cast<uint32_t>(h);
    return e;
}

// OR bits into a device error word from the host, as a kernel would.
cudaError_t or_error_word(int32_t *word, uint32_t bits) {
    int32_t h = 0;
    cudaError_t e = cudaMemcpy(&h, word, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    h |= static_cast<int32_t>(bits);
    e = cudaMemcpy(word, &h, sizeof h, cudaMemcpyHostToDevice);
    return e;
}

// The status of an error word's bits: a timeout leaves a tile's output
// unwritten, so it is reported first; the message names every bit set.
int error_status(uint32_t bits, const char *who) {
    if (bits == 0) return PKV_OK;
    const bool t = (bits & PKV_DEVERR_TIMEOUT) != 0, b = (bits & PKV_DEVERR_BOUNDS) != 0;
    if (t)
        return fail(PKV_ERR_DEVICE_TIMEOUT,
                    "%s gave up a bounded wait and left its tile unwritten%s", who,
                    b ? "; a kernel also met a block id or page index out of range" : "");
    return fail(PKV_ERR_DEVICE_BOUNDS, "%s met a block id or page index out of range and skipped it",
                who);
}

}  // namespace

// ================================================================== C ABI ====
extern "C" {

const char *pkv_last_error(void) { return g_last_error.c_str(); }

pkv_pool *pkv_pool_new(int32_t n_blocks, int32_t n_layers, int32_t kv_dim, int32_t block_size,
                       void *k_pool_dev, void *v_pool_dev, int32_t max_seqs,
                       int32_t max_blocks_per_seq, pkv_stream_t stream, uint32_t flags) {
    if (n_blocks <= 0 || n_layers <= 0 || kv_dim <= 0 || block_size <= 0 || max_seqs <= 0 ||
        max_blocks_per_seq <= 0) {
        fail(PKV_ERR_BAD_DIM, "pool sizes must be positive");
        return nullptr;
    }
    if (static_cast<int64_t>(max_seqs) * max_blocks_per_seq > (1LL << 31)) {
        fail(PKV_ERR_BAD_DIM, "max_seqs * max_blocks_per_seq too large");
        return nullptr;
    }
    auto *p = new pkv_pool();
    p->n_blocks = n_blocks;
    p->n_layers = n_layers;
    p->kv_dim = kv_dim;
    p->bs = block_size;
    p->bs_shift = (block_size & (block_size - 1)) == 0 ? __builtin_ctz(block_size) : -1;
    p->max_seqs = max_seqs;
    p->max_blocks = max_blocks_per_seq;
    p->host_only = (flags & PKV_POOL_HOST_ONLY) != 0;
    p->bf16 = (flags & PKV_POOL_BF16) != 0;
    p->fp8 = (flags & PKV_POOL_FP8) != 0;
    if (p->bf16 && p->fp8) {
        fail(PKV_ERR_ARG, "PKV_POOL_BF16 and PKV_POOL_FP8 exclude each other");
        delete p;
        return nullptr;
    }
    if (p->bf16 && (kv_dim % 2) != 0) {
        fail(PKV_ERR_BAD_DIM, "a bf16 pool needs an even kv_dim");
        delete p;
        return nullptr;
    }
    if (p->fp8 && (kv_dim % 4) != 0) {
        fail(PKV_ERR_BAD_DIM, "an fp8 pool needs kv_dim to be a multiple of 4");
        delete p;
        return nullptr;
    }
    p->free_stack.resize(n_blocks);
    for (int32_t i = 0; i < n_blocks; ++i) p->free_stack[i] = n_blocks - 1 - i;
    p->refcnt.assign(n_blocks, 0);
    p->free_slots.resize(max_seqs);
    for (int32_t i = 0; i < max_seqs; ++i) p->free_slots[i] = max_seqs - 1 - i;
    p->slot_owner.assign(max_seqs, nullptr);
    if (p->host_only) return p;

    p->stream = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->n_sm, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) {
        cuda_fail(e, "cudaGetDevice");
        delete p;
        return nullptr;
    }
    if ((k_pool_dev == nullptr) != (v_pool_dev == nullptr)) {
        fail(PKV_ERR_ARG, "pass both K and V pool buffers or neither");
        delete p;
        return nullptr;
    }
    const size_t pool_bytes = static_cast<size_t>(n_blocks) * p->block_floats() * p->elem_bytes();
    if (k_pool_dev) {
        if (!aligned16(k_pool_dev) || !aligned16(v_pool_dev)) {
            fail(PKV_ERR_ARG, "pool buffers must be 16-byte aligned");
            delete p;
            return nullptr;
        }
        p->k = k_pool_dev;
        p->v = v_pool_dev;
    } else {
        e = cudaMalloc(&p->k, pool_bytes);
        if (e == cudaSuccess) e = cudaMalloc(&p->v, pool_bytes);
        if (e != cudaSuccess) {
            cuda_fail(e, "pool allocation");
            cudaFree(p->k);
            delete p;
            return nullptr;
        }
        p->owns_kv = true;
    }
    e = cudaMalloc(&p->pt_dev, static_cast<size_t>(max_seqs) * max_blocks_per_seq * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMalloc(&p->err_dev, sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMemsetAsync(p->pt_dev, 0xff, static_cast<size_t>(max_seqs) * max_blocks_per_seq * sizeof(int32_t),
                            p->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->err_dev, 0, sizeof(int32_t), p->stream);
    if (e != cudaSuccess) {
        cuda_fail(e, "pool metadata allocation");
        pkv_pool_free(p);
        return nullptr;
    }
    return p;
}

void pkv_pool_free(pkv_pool *p) {
    if (!p) return;
    for (pkv_seq *s : p->slot_owner) delete s;
    p->slot_owner.clear();
    if (!p->host_only) {
        DevGuard dg(p->device);
        p->desc.release(p->stream);
        p->part.release(p->stream);
        p->io_in.release(p->stream);
        p->io_out.release(p->stream);
        p->qrot.release(p->stream);
        p->img.release(p->stream);
        p->icache.buf.release(p->stream);
        cudaStreamSynchronize(p->stream);
        p->stager.destroy();

        if (p->owns_kv) {
            cudaFree(p->k);
            cudaFree(p->v);
        }
        cudaFree(p->pt_dev);
        cudaFree(p->err_dev);
    }
    delete p;
}

int pkv_pool_set_image_cache(pkv_pool *p, int64_t max_bytes) {
    if (!p || p->host_only) return fail(PKV_ERR_ARG, "image cache needs a device pool");
    if (max_bytes < 0) return fail(PKV_ERR_ARG, "negative image cache size");
    DevGuard dg(p->device);
    ImageCache &ic = p->icache;
    // one slot: a 64-key tile's images for every kv head of head_dim 128
    const size_t slot_bytes = static_cast<size_t>(ceil_div(p->kv_dim, 128)) * kImageBytes;
    const int64_t n = max_bytes / static_cast<int64_t>(slot_bytes);
    ic.reset(0);
    ic.buf.release(p->stream);
    if (n <= 0) {
        p->gen.clear();
        p->gen.shrink_to_fit();
        return PKV_OK;
    }
    if (n > 0x7fffffffLL) return fail(PKV_ERR_ARG, "image cache too large");
    cudaError_t e = ic.buf.ensure(static_cast<size_t>(n) * slot_bytes, p->stream, p->device);
    if (e != cudaSuccess) {
        ic.buf.release(p->stream);
        return cuda_fail(e, "image cache buffer");
    }
    // generations start over: nothing cached depends on earlier ones
    p->gen.assign(static_cast<size_t>(p->n_blocks) * p->n_layers, 0u);
    ic.slot_bytes = slot_bytes;
    ic.reset(static_cast<int32_t>(n));
    return PKV_OK;
}

int pkv_pool_set_stream(pkv_pool *p, pkv_stream_t stream) {
    if (!p) return fail(PKV_ERR_ARG, "NULL pool");
    p->stream = static_cast<cudaStream_t>(stream);
    return PKV_OK;
}

void *pkv_pool_k_data(const pkv_pool *p) { return p ? p->k : nullptr; }
void *pkv_pool_v_data(const pkv_pool *p) { return p ? p->v : nullptr; }
int pkv_pool_set_kv_scale(pkv_pool *p, float scale) {
    if (!p) return fail(PKV_ERR_ARG, "NULL pool");
    if (!p->fp8) return fail(PKV_ERR_ARG, "the scale applies to fp8 pools only");
    int ex = 0;
    const float m = std::frexp(scale, &ex);
    if (!(scale > 0.f) || m != 0.5f || ex < -19 || ex > 21)
        return fail(PKV_ERR_ARG, "the scale must be a power of two in [2^-20, 2^20]");
    if (static_cast<int32_t>(p->free_stack.size()) != p->n_blocks)
        return fail(PKV_ERR_ARG, "the scale can only change while no block is in use");
    p->kv_scale = scale;
    return PKV_OK;
}

int pkv_pool_last_work(const pkv_pool *p, int64_t *out, int32_t cap) {
    if (!p || !out || cap < 0) return fail(PKV_ERR_ARG, "NULL pool or output");
    const int32_t n = std::min<int32_t>(cap, PKV_WORK_FIELDS);
    std::copy(p->last_work, p->last_work + n, out);
    return PKV_OK;
}

int32_t pkv_pool_free_blocks(const pkv_pool *p) {
    return p ? static_cast<int32_t>(p->free_stack.size()) : -1;
}

int64_t pkv_alloc_block(pkv_pool *p) {
    if (!p) {
        fail(PKV_ERR_ARG, "NULL pool");
        return -1;
    }
    int32_t b = pop_block(p);
    if (b < 0) fail(PKV_ERR_EXHAUSTED, "pool exhausted");
    return b;
}

int pkv_unref_block(pkv_pool *p, int64_t id) {
    if (!p) return fail(PKV_ERR_ARG, "NULL pool");
    if (id < 0 || id >= p->n_blocks || p->refcnt[id] <= 0)
        return fail(PKV_ERR_ARG, "block %lld is not allocated", static_cast<long long>(id));
    unref(p, static_cast<int32_t>(id));
    return PKV_OK;
}

int32_t pkv_refcnt(const pkv_pool *p, int64_t id) {
    if (!p || id < 0 || id >= p->n_blocks) return -1;
    return p->refcnt[id];
}

pkv_seq *pkv_seq_new(pkv_pool *p, int32_t max_tokens) {
    if (!p) {
        fail(PKV_ERR_ARG, "NULL pool");
        return nullptr;
    }
    if (max_tokens <= 0 || ceil_div(max_tokens, p->bs) > p->max_blocks) {
        fail(PKV_ERR_CAPACITY, "max_tokens %d outside (0, %lld]", max_tokens,
             static_cast<long long>(p->max_blocks) * p->bs);
        return nullptr;
    }
    if (p->free_slots.empty()) {
        fail(PKV_ERR_CAPACITY, "max_seqs sequences are live");
        return nullptr;
    }
    auto *s = new pkv_seq();
    s->pool = p;
    s->slot = p->free_slots.back();
    p->free_slots.pop_back();
    s->max_tokens = max_tokens;
    p->slot_owner[s->slot] = s;
    return s;
}

pkv_seq *pkv_seq_fork(pkv_seq *parent) {
    if (!parent) {
        fail(PKV_ERR_SEQ, "NULL sequence");
        return nullptr;
    }
    pkv_pool *p = parent->pool;
    if (p->free_slots.empty()) {
        fail(PKV_ERR_CAPACITY, "max_seqs sequences are live");
        return nullptr;
    }
    auto *s = new pkv_seq();
    s->pool = p;
    s->slot = p->free_slots.back();
    p->free_slots.pop_back();
    s->max_tokens = parent->max_tokens;
    s->len = parent->len;
    s->pt = parent->pt;
    for (int32_t b : s->pt) p->refcnt[b] += 1;
    p->slot_owner[s->slot] = s;
    mark_dirty(s, 0, static_cast<int32_t>(s->pt.size()));
    return s;
}

int pkv_seq_free(pkv_seq *s) {
    if (!s) return fail(PKV_ERR_ARG, "NULL sequence");
    pkv_pool *p = s->pool;
    for (auto it = s->pt.rbegin(); it != s->pt.rend(); ++it) unref(p, *it);
    if (s->dirty) p->dirty.erase(std::remove(p->dirty.begin(), p->dirty.end(), s), p->dirty.end());
    p->slot_owner[s->slot] = nullptr;
    p->free_slots.push_back(s->slot);
    delete s;
    return PKV_OK;
}

int pkv_seq_truncate(pkv_seq *s, int32_t new_len) {
    if (!s) return fail(PKV_ERR_ARG, "NULL sequence");
    if (new_len < 0 || new_len > s->len)
        return fail(PKV_ERR_ARG, "truncate to %d outside [0, %d]", new_len, s->len);
    pkv_pool *p = s->pool;
    const int32_t keep = ceil_div(new_len, p->bs);
    for (int32_t k = static_cast<int32_t>(s->pt.size()) - 1; k >= keep; --k) unref(p, s->pt[k]);
    if (static_cast<int32_t>(s->pt.size()) > keep) s->pt.resize(keep);
    s->len = new_len;
    return PKV_OK;
}

int pkv_seq_truncate_batch(pkv_seq *const *seqs, int32_t M, const int32_t *new_len) {
    if (M <= 0 || !seqs || !new_len) return fail(PKV_ERR_ARG, "empty batch");
    for (int32_t r = 0; r < M; ++r)
        if (!seqs[r]) return fail(PKV_ERR_ARG, "sequence %d is NULL", r);
    pkv_pool *p = seqs[0]->pool;
    for (int32_t r = 1; r < M; ++r)
        if (seqs[r]->pool != p) return fail(PKV_ERR_ARG, "sequences of different pools in one batch");
    {
        int rc = check_dup(p, seqs, M);
        if (rc) return rc;
    }
    for (int32_t r = 0; r < M; ++r)
        if (new_len[r] < 0 || new_len[r] > seqs[r]->len)
            return fail(PKV_ERR_ARG, "row %d: truncate to %d outside [0, %d]", r, new_len[r], seqs[r]->len);
    for (int32_t r = 0; r < M; ++r) pkv_seq_truncate(seqs[r], new_len[r]);
    return PKV_OK;
}

int32_t pkv_seq_len(const pkv_seq *s) { return s ? s->len : -1; }
int32_t pkv_seq_slot(const pkv_seq *s) { return s ? s->slot : -1; }

int32_t pkv_seq_page_table(const pkv_seq *s, int32_t *out, int32_t cap) {
    if (!s) return -1;
    const int32_t n = static_cast<int32_t>(s->pt.size());
    if (out)
        for (int32_t i = 0; i < std::min(n, cap); ++i) out[i] = s->pt[i];
    return n;
}

int pkv_ensure_append_batch(pkv_seq *const *seqs, int32_t M, const int32_t *n) {
    if (M <= 0 || !seqs || !n) return fail(PKV_ERR_ARG, "empty batch");
    for (int32_t r = 0; r < M; ++r)
        if (!seqs[r]) return fail(PKV_ERR_ARG, "sequence %d is NULL", r);
    pkv_pool *p = seqs[0]->pool;
    for (int32_t r = 1; r < M; ++r)
        if (seqs[r]->pool != p) return fail(PKV_ERR_ARG, "sequences of different pools in one batch");
    {
        int rc = check_dup(p, seqs, M);
        if (rc) return rc;
    }
    // pass 1: validate row by row and count blocks, as the rows would consume
    // them in order (a block shared by two rows is copied by the first only)
    std::unordered_map<int32_t, int32_t> dec;
    int64_t needed = 0;
    const int64_t avail = static_cast<int64_t>(p->free_stack.size());
    for (int32_t r = 0; r < M; ++r) {
        const pkv_seq *s = seqs[r];
        if (n[r] <= 0) return fail(PKV_ERR_ARG, "n[%d] = %d must be positive", r, n[r]);
        if (static_cast<int64_t>(s->len) + n[r] > s->max_tokens)
            return fail(PKV_ERR_CAPACITY, "row %d: len %d + %d exceeds max_tokens %d", r, s->len, n[r],
                        s->max_tokens);
        const int32_t first = s->len / p->bs;
        const int32_t last = (s->len + n[r] - 1) / p->bs;
        const int32_t have = static_cast<int32_t>(s->pt.size());
        for (int32_t k = first; k <= last && k < have; ++k) {
            const int32_t b = s->pt[k];
            auto it = dec.find(b);
            const int32_t eff = p->refcnt[b] - (it == dec.end() ? 0 : it->second);
            if (eff > 1) {
                ++needed;
                ++dec[b];
            }
        }
        needed += std::max(0, last + 1 - have);
        if (needed > avail)
            return fail(PKV_ERR_EXHAUSTED, "pool exhausted (%lld blocks needed, %lld free)",
                        static_cast<long long>(needed), static_cast<long long>(avail));
    }
    // pass 2: apply
    std::vector<CopyDesc> copies;
    for (int32_t r = 0; r < M; ++r) {
        pkv_seq *s = seqs[r];
        const int32_t first = s->len / p->bs;
        const int32_t last = (s->len + n[r] - 1) / p->bs;
        const int32_t have = static_cast<int32_t>(s->pt.size());
        for (int32_t k = first; k <= last && k < have; ++k) {
            const int32_t b = s->pt[k];
            if (p->refcnt[b] > 1) {
                const int32_t nb = pop_block(p);
                copies.push_back({b, nb});
                unref(p, b);
                s->pt[k] = nb;
                mark_dirty(s, k, k + 1);
            }
        }
        for (int32_t k = have; k <= last; ++k) s->pt.push_back(pop_block(p));
        mark_dirty(s, have, last + 1);
    }
    if (copies.empty() || p->host_only) return PKV_OK;

    DevGuard dg(p->device);
    p->blob.clear();
    const size_t off = p->blob.put(copies.data(), copies.size());
    cudaError_t e = upload_blob(p);
    if (e != cudaSuccess) return cuda_fail(e, "copy list upload");
    e = launch(PKV_KERNEL_COPY, p->stream, [&] {
        return launch_copy_blocks(p->k, p->v, dptr<CopyDesc>(p, off), static_cast<int32_t>(copies.size()),
                                  p->block_floats() * static_cast<int64_t>(p->elem_bytes()) / 4,
                                  p->n_blocks, p->err_dev, p->stream);
    });
    if (e != cudaSuccess) return cuda_fail(e, "copy-on-append kernel");
    return PKV_OK;
}

int pkv_ensure_append(pkv_seq *s, int32_t n) { return pkv_ensure_append_batch(&s, 1, &n); }

int pkv_advance_batch(pkv_seq *const *seqs, int32_t M, const int32_t *n) {
    if (M <= 0 || !seqs || !n) return fail(PKV_ERR_ARG, "empty batch");
    for (int32_t r = 0; r < M; ++r)
        if (!seqs[r]) return fail(PKV_ERR_ARG, "sequence %d is NULL", r);
    pkv_pool *p = seqs[0]->pool;
    for (int32_t r = 1; r < M; ++r)
        if (seqs[r]->pool != p) return fail(PKV_ERR_ARG, "sequences of different pools in one batch");
    {
        int rc = check_dup(p, seqs, M);
        if (rc) return rc;
    }
    for (int32_t r = 0; r < M; ++r) {
        const pkv_seq *s = seqs[r];
        if (n[r] <= 0) return fail(PKV_ERR_ARG, "n[%d] = %d must be positive", r, n[r]);
        if (static_cast<int64_t>(s->len) + n[r] > s->max_tokens)
            return fail(PKV_ERR_CAPACITY, "row %d: advance past max_tokens", r);
        if (static_cast<int64_t>(s->len) + n[r] > static_cast<int64_t>(s->pt.size()) * p->bs)
            return fail(PKV_ERR_SEQ, "row %d: advance past the ensured blocks", r);
    }
    for (int32_t r = 0; r < M; ++r) seqs[r]->len += n[r];
    return PKV_OK;
}

int pkv_advance(pkv_seq *s, int32_t n) { return pkv_advance_batch(&s, 1, &n); }

int pkv_append_layer(pkv_seq *seq, int32_t layer, const float *K_new, const float *V_new,
                     int32_t n_tokens) {
    return run_layer(&seq, 1, &n_tokens, nullptr, K_new, V_new, 0, 0, 0, layer, 0, 0.f, nullptr,
                     false, false);
}

int pkv_attn_with_paged(const float *Q, const float *K_new, const float *V_new, int32_t n_tokens,
                        int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, pkv_seq *seq,
                        int32_t layer, int32_t causal, float scale, float *out) {
    if (n_tokens <= 0) return fail(PKV_ERR_BAD_DIM, "n_tokens must be positive");
    return run_layer(&seq, 1, &n_tokens, Q, K_new, V_new, n_heads, n_kv_heads, head_dim, layer,
                     causal, scale, out, false, true);
}

int pkv_attn_batch(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q,
                   const float *K_new, const float *V_new, int32_t n_heads, int32_t n_kv_heads,
                   int32_t head_dim, int32_t layer, int32_t causal, float scale, float *out) {
    return run_layer(seqs, M, n_q, Q, K_new, V_new, n_heads, n_kv_heads, head_dim, layer, causal,
                     scale, out, false, true);
}

int pkv_attn_batch_rope(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q,
                        const float *K_new, const float *V_new, int32_t n_heads, int32_t n_kv_heads,
                        int32_t head_dim, int32_t layer, int32_t causal, float scale,
                        double rope_base, float *out) {
    if (!(rope_base > 0.0)) return fail(PKV_ERR_ARG, "RoPE base must be positive");
    return run_layer(seqs, M, n_q, Q, K_new, V_new, n_heads, n_kv_heads, head_dim, layer, causal,
                     scale, out, false, true, rope_base);
}

int pkv_attn_batch_host(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q_host,
                        const float *K_new_host, const float *V_new_host, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, int32_t layer, int32_t causal,
                        float scale, float *out_host) {
    return run_layer_host(seqs, M, n_q, Q_host, K_new_host, V_new_host, n_heads, n_kv_heads,
                          head_dim, layer, causal, scale, out_host);
}

int pkv_attn_contiguous(const float *Q, const float *Kc, const float *Vc, int32_t n_q,
                        int32_t total_k, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                        int32_t causal, float scale, float *out, pkv_stream_t stream) {
    if (n_q <= 0) return fail(PKV_ERR_BAD_DIM, "n_q must be positive");
    int rc = check_heads(n_heads, n_kv_heads, head_dim);
    if (rc) return rc;
    if (total_k < n_q) return fail(PKV_ERR_BAD_DIM, "total_k %d < n_q %d", total_k, n_q);
    if (head_dim > kMaxHeadDim)
        return fail(PKV_ERR_BAD_DIM, "head_dim %d > %d is not supported", head_dim, kMaxHeadDim);
    if (!Q || !Kc || !Vc || !out) return fail(PKV_ERR_ARG, "NULL data pointer");
    if ((head_dim % 4) == 0 ? (!aligned16(Q) || !aligned16(Kc) || !aligned16(Vc) || !aligned16(out))
                            : (!aligned4(Q) || !aligned4(Kc) || !aligned4(Vc) || !aligned4(out)))
        return fail(PKV_ERR_ARG, "device pointers must be 16-byte aligned (4-byte if head_dim %% 4 != 0)");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PKV_ERR_ARG, "device index out of range");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    std::vector<RowDesc> rows{{0, total_k - n_q, n_q, 0}};
    WorkList w;
    const int32_t S = g_split_keys.load();
    build_work(rows, causal, S, head_dim, n_heads / n_kv_heads, w);
    // the tensor-core tiles' operand images: every 64-key tile of the row
    std::vector<SplitItem> items;
    std::vector<int32_t> img_tile0, img_slot;
    if (!w.tiles.empty()) {
        const int32_t nt = ceil_div(total_k, kKeyTile);
        img_tile0.push_back(0);
        for (int32_t kt = 0; kt < nt; ++kt) {
            img_slot.push_back(kt);
            items.push_back({0, kt, kt});
        }
    }
    Blob blob;
    const size_t rows_off = blob.put(rows.data(), 1);
    const size_t units_off = blob.put(w.units.data(), w.units.size());
    const size_t tiles_off = blob.put(w.tiles.data(), w.tiles.size());
    const size_t merges_off = blob.put(w.merges.data(), w.merges.size());
    const size_t items_off = blob.put(items.data(), items.size());
    const size_t tile0_off = blob.put(img_tile0.data(), img_tile0.size());
    const size_t slot_off = blob.put(img_slot.data(), img_slot.size());
    const size_t desc_bytes = (blob.size() + 255) & ~static_cast<size_t>(255);
    const size_t pf = static_cast<size_t>(w.n_part) * n_heads;
    const size_t part_bytes = (pf * (2 + head_dim) * sizeof(float) + 255) & ~static_cast<size_t>(255);
    const size_t img_bytes = img_slot.size() * static_cast<size_t>(n_kv_heads) * kImageBytes;
    const size_t total = desc_bytes + part_bytes + img_bytes;

    std::lock_guard<std::mutex> lk(g_contig_mu);
    int32_t *err_word = nullptr;
    e = contig_error_word(dev, &err_word);
    if (e != cudaSuccess) return cuda_fail(e, "error word");
    cudaMemPool_t mp;
    e = mempool_for(dev, &mp);
    if (e != cudaSuccess) return cuda_fail(e, "memory pool");
    void *mem = nullptr;
    e = cudaMallocFromPoolAsync(&mem, total, mp, st);
    if (e != cudaSuccess) return cuda_fail(e, "scratch allocation");
    unsigned char *base = static_cast<unsigned char *>(mem);
    e = g_contig_stager[dev].upload(base, blob.b.data(), blob.b.size(), st);
    if (e != cudaSuccess) {
        cudaFreeAsync(mem, st);
        return cuda_fail(e, "descriptor upload");
    }
    AttnArgs a{};
    a.Q = Q;
    a.out = out;
    a.rows = reinterpret_cast<const RowDesc *>(base + rows_off);
    a.units = reinterpret_cast<const UnitDesc *>(base + units_off);
    a.merges = reinterpret_cast<const MergeDesc *>(base + merges_off);
    a.n_units = static_cast<int32_t>(w.units.size());
    a.n_heads = n_heads;
    a.n_kv = n_kv_heads;
    a.hd = head_dim;
    a.group = n_heads / n_kv_heads;
    a.causal = causal ? 1 : 0;
    a.split_keys = S;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.err = err_word;
    if (pf > 0) {
        a.pm = reinterpret_cast<float *>(base + desc_bytes);
        a.pl = a.pm + pf;
        a.pacc = a.pl + pf;
    }
    const ContigAddr addr{Kc, Vc, n_kv_heads * head_dim};
    if (!w.tiles.empty()) {
        unsigned char *img = base + desc_bytes + part_bytes;
        const SplitArgs sa{a.rows, reinterpret_cast<const SplitItem *>(base + items_off),
                           static_cast<int32_t>(items.size()), n_kv_heads, img, a.err};
        e = launch(PKV_KERNEL_SPLIT, st, [&] { return launch_split_contig(sa, addr, st); });
        PrefillArgs pa{Q, out, a.rows, reinterpret_cast<const PrefillTile *>(base + tiles_off),
                       static_cast<int32_t>(w.tiles.size()), a.pm, a.pl, a.pacc, n_heads,
                       n_kv_heads, a.group, a.causal, S * kPrefillSplitFactor, a.scale_log2,
                       a.err};
        pa.img = img;
        pa.img_tile0 = reinterpret_cast<const int32_t *>(base + tile0_off);
        pa.img_slot = reinterpret_cast<const int32_t *>(base + slot_off);
        if (e == cudaSuccess)
            e = launch(PKV_KERNEL_PREFILL, st, [&] { return launch_prefill_contig(pa, addr, st); });
    }
    if (e == cudaSuccess && !w.units.empty())
        e = launch(PKV_KERNEL_DECODE, st, [&] { return launch_decode_contig(a, addr, st); });
    if (e == cudaSuccess && !w.merges.empty()) {
        MergeArgs m{a.pm, a.pl, a.pacc, out, a.rows,
                    reinterpret_cast<const MergeDesc *>(base + merges_off),
                    static_cast<int32_t>(w.merges.size()), n_heads, head_dim};
        e = launch(PKV_KERNEL_MERGE, st, [&] { return launch_merge(m, st); });
    }
    cudaFreeAsync(mem, st);
    if (e != cudaSuccess) return cuda_fail(e, "contiguous attention kernels");
    return PKV_OK;
}

int pkv_sync_error(pkv_pool *p) {
    if (!p) return fail(PKV_ERR_ARG, "NULL pool");
    if (p->host_only) return PKV_OK;
    DevGuard dg(p->device);
    cudaError_t e = cudaStreamSynchronize(p->stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    uint32_t h = 0;
    e = take_error_word(p->err_dev, &h);
    if (e != cudaSuccess) return cuda_fail(e, "error word");
    return error_status(h, "a pool kernel");
}

int pkv_contiguous_sync_error(pkv_stream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PKV_ERR_ARG, "device index out of range");
    e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    uint32_t h = 0, hn = 0;
    {
        std::lock_guard<std::mutex> lk(g_contig_mu);
        e = take_error_word(g_contig_err[dev], &h);
    }
    if (e == cudaSuccess) e = take_error_word(noalloc_error_word(dev, false, nullptr), &hn);
    if (e != cudaSuccess) return cuda_fail(e, "error word");
    return error_status(h | hn, "a contiguous-path kernel");
}

int pkv_debug_or_error_bits(pkv_pool *p, int32_t which, uint32_t bits) {
    if ((bits & ~(PKV_DEVERR_BOUNDS | PKV_DEVERR_TIMEOUT)) != 0)
        return fail(PKV_ERR_ARG, "bits 0x%x outside PKV_DEVERR_*", bits);
    int32_t *word = nullptr;
    cudaError_t e = cudaSuccess;
    if (which == PKV_ERRWORD_POOL) {
        if (!p || p->host_only) return fail(PKV_ERR_ARG, "a device pool is needed");
        DevGuard dg(p->device);
        e = cudaStreamSynchronize(p->stream);
        if (e == cudaSuccess) e = or_error_word(p->err_dev, bits);
        if (e != cudaSuccess) return cuda_fail(e, "error word");
        return PKV_OK;
    }
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PKV_ERR_ARG, "device index out of range");
    if (which == PKV_ERRWORD_CONTIGUOUS) {
        std::lock_guard<std::mutex> lk(g_contig_mu);
        e = contig_error_word(dev, &word);
        if (e == cudaSuccess) e = or_error_word(word, bits);
    } else if (which == PKV_ERRWORD_NOALLOC) {
        word = noalloc_error_word(dev, true, &e);
        if (e == cudaSuccess) e = or_error_word(word, bits);
    } else {
        return fail(PKV_ERR_ARG, "unknown error word %d", which);
    }
    if (e != cudaSuccess) return cuda_fail(e, "error word");
    return PKV_OK;
}

int pkv_pool_flush(pkv_pool *p) {
    if (!p) return fail(PKV_ERR_ARG, "NULL pool");
    if (p->host_only || p->dirty.empty()) return PKV_OK;
    DevGuard dg(p->device);
    p->blob.clear();
    size_t runs_off, vals_off;
    int32_t n_runs;
    put_pt_runs(p, p->blob, &runs_off, &n_runs, &vals_off);
    if (n_runs == 0) return PKV_OK;
    cudaError_t e = upload_blob(p);
    if (e != cudaSuccess) return cuda_fail(e, "page-table upload");
    e = launch(PKV_KERNEL_PAGETABLE, p->stream, [&] {
        return launch_pt_apply(p->pt_dev, p->max_blocks, dptr<PtRun>(p, runs_off), n_runs,
                               dptr<int32_t>(p, vals_off), p->stream);
    });
    if (e != cudaSuccess) return cuda_fail(e, "page-table upload kernel");
    return PKV_OK;
}

int pkv_set_split_keys(int32_t keys) {
    if (keys < 32 || keys > 65536 || (keys % 32) != 0)
        return fail(PKV_ERR_ARG, "split keys %d: need a multiple of 32 in [32, 65536]", keys);
    g_split_keys.store(keys);
    return PKV_OK;
}
int32_t pkv_get_split_keys(void) { return g_split_keys.load(); }

int pkv_set_fused_append(int32_t on) {
    g_fused_append.store(on ? 1 : 0);
    return PKV_OK;
}
int32_t pkv_get_fused_append(void) { return g_fused_append.load(); }

int pkv_set_cascade(int32_t on) {
    g_cascade.store(on ? 1 : 0);
    return PKV_OK;
}
int32_t pkv_get_cascade(void) { return g_cascade.load(); }

int pkv_set_prefill_pairing(int32_t mode) {
    if (mode < 0 || mode > 2) return fail(PKV_ERR_ARG, "prefill pairing mode must be 0, 1 or 2");
    g_prefill_pairing.store(mode);
    return PKV_OK;
}
int32_t pkv_get_prefill_pairing(void) { return g_prefill_pairing.load(); }

int64_t pkv_launch_count(void) { return g_launches.load(); }

int pkv_profile_enable(int32_t on) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.on = on != 0;
    return PKV_OK;
}

int pkv_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.drain();
    for (int k = 0; k < PKV_KERNEL_KINDS; ++k) {
        g_prof.ms[k] = 0;
        g_prof.n[k] = 0;
    }
    return PKV_OK;
}

int pkv_profile_read(int32_t kind, double *ms, int64_t *launches) {
    if (kind < 0 || kind >= PKV_KERNEL_KINDS) return fail(PKV_ERR_ARG, "kernel kind %d", kind);
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.drain();
    if (ms) *ms = g_prof.ms[kind];
    if (launches) *launches = g_prof.n[kind];
    return PKV_OK;
}

}  // extern "C"

// ------------------------------------------- helpers for other entry points ----
namespace pkv {

void build_contig_work(int32_t n_q, int32_t total_k, int32_t causal, int32_t split_keys,
                       int32_t head_dim, int32_t group, std::vector<UnitDesc> &units,
                       std::vector<PrefillTile> &tiles, std::vector<MergeDesc> &merges,
                       int64_t *n_part, bool allow_tc) {
    WorkList w;
    std::vector<RowDesc> rows{{0, total_k - n_q, n_q, 0}};
    build_work(rows, causal, split_keys, head_dim, group, w, {}, 0, 0, allow_tc);
    units.swap(w.units);
    tiles.swap(w.tiles);
    merges.swap(w.merges);
    *n_part = w.n_part;
}

cudaError_t launch_counted(int kind, cudaStream_t s, cudaError_t (*fn)(void *), void *ctx) {
    return launch(kind, s, [&] { return fn(ctx); });
}

int32_t current_split_keys() { return g_split_keys.load(); }

int report_error(int code, const char *msg) { return fail(code, "%s", msg); }

}  // namespace pkv
