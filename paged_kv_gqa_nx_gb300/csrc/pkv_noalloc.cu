// pkv_noalloc.cu -- contiguous attention that allocates nothing.
//
// pkv_attn_contiguous obtains its per-call scratch (the work-list descriptor
// and the split-K partials) from a stream-ordered device memory pool.  Some
// callers cannot let a library allocate device memory: a serving engine that
// reserves its whole device-memory budget up front (a further cudaMalloc
// would fail or break its accounting), code running inside an allocator or
// memory-pressure callback (allocating again would re-enter that allocator),
// and latency-critical loops where cudaMalloc / cudaFree may synchronise the
// device.  pkv_attn_contiguous_noalloc serves them: the same kernels, with the
// scratch in one file-scope device array that every GPU loading the library
// holds until the process exits.  A row of 32 or more queries takes the
// tensor-core kernel when its operand images (64 KiB per 64-key tile and kv
// head) fit in the array beside the rest, else the split-K decode kernels.
//
// The array's name is a host-side stand-in in host code, not a device
// address, so the entry point looks the address up once per device with
// cudaGetSymbolAddress (with that device current) and passes it to the
// kernels.  Every call shares the array and it keeps the previous call's
// contents.  Its first word is the kernels' error word: cleared once, when
// the device is set up, it gathers the bits of every call until
// pkv_contiguous_sync_error reads and clears it; everything else is fully
// written by a call before that call reads it.
#include "../../include/pkv.h"
#include "pkv_internal.h"

#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

using namespace pkv;

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;                     // serialises set-up and enqueueing on the host
void *g_scratch_dev[64] = {};        // device address of g_noalloc_scratch, per device

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct DecodeCtx {
    const AttnArgs *a;
    const ContigAddr *addr;
    cudaStream_t s;
};
cudaError_t run_decode(void *p) {
    auto *c = static_cast<DecodeCtx *>(p);
    return launch_decode_contig(*c->a, *c->addr, c->s);
}
struct PrefillCtx {
    const PrefillArgs *a;
    const ContigAddr *addr;
    cudaStream_t s;
};
cudaError_t run_prefill(void *p) {
    auto *c = static_cast<PrefillCtx *>(p);
    return launch_prefill_contig(*c->a, *c->addr, c->s);
}
struct SplitCtx {
    const SplitArgs *a;
    const ContigAddr *addr;
    cudaStream_t s;
};
cudaError_t run_split(void *p) {
    auto *c = static_cast<SplitCtx *>(p);
    return launch_split_contig(*c->a, *c->addr, c->s);
}
struct MergeCtx {
    const MergeArgs *m;
    cudaStream_t s;
};
cudaError_t run_merge(void *p) {
    auto *c = static_cast<MergeCtx *>(p);
    return launch_merge(*c->m, c->s);
}

int err_arg(int code, const char *msg) { return report_error(code, msg); }

// First use on device `dev` (current; g_mu held): look up the array's device
// address and clear its error word.  The clear is finished before this
// returns, so no stream needs ordering after it.
cudaError_t set_up(int dev) {
    if (g_scratch_dev[dev]) return cudaSuccess;
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaSuccess && !p) e = cudaErrorInvalidSymbol;
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = p;
    return cudaSuccess;
}

}  // namespace

namespace pkv {

int32_t *noalloc_error_word(int dev, bool setup, cudaError_t *e) {
    if (e) *e = cudaSuccess;
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_dev[dev] && setup) {
        const cudaError_t r = set_up(dev);
        if (r != cudaSuccess) {
            if (e) *e = r;
            return nullptr;
        }
    }
    return static_cast<int32_t *>(g_scratch_dev[dev]);
}

}  // namespace pkv

extern "C" int pkv_attn_contiguous_noalloc(const float *Q, const float *Kc, const float *Vc,
                                           int32_t n_q, int32_t total_k, int32_t n_heads,
                                           int32_t n_kv_heads, int32_t head_dim, int32_t causal,
                                           float scale, float *out, pkv_stream_t stream) {
    if (n_q <= 0) return err_arg(PKV_ERR_BAD_DIM, "n_q must be positive");
    if (n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return err_arg(PKV_ERR_BAD_DIM, "n_heads, n_kv_heads and head_dim must be positive");
    if (n_heads % n_kv_heads != 0)
        return err_arg(PKV_ERR_BAD_GQA, "n_heads is not a multiple of n_kv_heads");
    if (total_k < n_q) return err_arg(PKV_ERR_BAD_DIM, "total_k < n_q");
    if (head_dim > kMaxHeadDim) return err_arg(PKV_ERR_BAD_DIM, "head_dim > 256 is not supported");
    if (!Q || !Kc || !Vc || !out) return err_arg(PKV_ERR_ARG, "NULL data pointer");
    const uintptr_t mask = (head_dim % 4) == 0 ? 15 : 3;
    if (((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(Kc) |
          reinterpret_cast<uintptr_t>(Vc) | reinterpret_cast<uintptr_t>(out)) & mask) != 0)
        return err_arg(PKV_ERR_ARG, "device pointers must be 16-byte aligned (4-byte if head_dim % 4 != 0)");

    // work list and the scratch layout:
    // [error word][rows][units][tiles][merges][items][image lists][partials][images]
    const int32_t S = current_split_keys();
    std::vector<UnitDesc> units;
    std::vector<PrefillTile> tiles;
    std::vector<MergeDesc> merges;
    std::vector<SplitItem> items;
    std::vector<int32_t> img_tile0, img_slot;
    int64_t n_part = 0;
    const RowDesc row{0, total_k - n_q, n_q, 0};
    size_t rows_off = 0, units_off = 0, tiles_off = 0, merges_off = 0, items_off = 0, tile0_off = 0,
           slot_off = 0, desc_end = 0, part_off = 0, img_off = 0, pf = 0, total = 0;
    auto lay_out = [&](bool allow_tc) {
        build_contig_work(n_q, total_k, causal, S, head_dim, n_heads / n_kv_heads, units, tiles, merges,
                          &n_part, allow_tc);
        items.clear();
        img_tile0.clear();
        img_slot.clear();
        if (!tiles.empty()) {
            // the tensor-core tiles' operand images: every 64-key tile of the row
            const int32_t nt = (total_k + kKeyTile - 1) / kKeyTile;
            img_tile0.push_back(0);
            for (int32_t kt = 0; kt < nt; ++kt) {
                img_slot.push_back(kt);
                items.push_back({0, kt, kt});
            }
        }
        rows_off = 256;
        units_off = round256(rows_off + sizeof(RowDesc));
        tiles_off = round256(units_off + units.size() * sizeof(UnitDesc));
        merges_off = round256(tiles_off + tiles.size() * sizeof(PrefillTile));
        items_off = round256(merges_off + merges.size() * sizeof(MergeDesc));
        tile0_off = round256(items_off + items.size() * sizeof(SplitItem));
        slot_off = round256(tile0_off + img_tile0.size() * sizeof(int32_t));
        desc_end = round256(slot_off + img_slot.size() * sizeof(int32_t));
        part_off = desc_end;
        pf = static_cast<size_t>(n_part) * n_heads;
        img_off = round256(part_off + pf * (2 + static_cast<size_t>(head_dim)) * sizeof(float));
        total = img_off + img_slot.size() * static_cast<size_t>(n_kv_heads) * kImageBytes;
    };
    lay_out(true);
    if (total > kScratchBytes && !tiles.empty()) lay_out(false);  // the images do not fit
    if (total > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "request needs %zu bytes of scratch, more than the %zu-byte static array of "
                 "pkv_attn_contiguous_noalloc; use pkv_attn_contiguous",
                 total, kScratchBytes);
        return err_arg(PKV_ERR_CAPACITY, msg);
    }

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return err_arg(PKV_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return err_arg(PKV_ERR_ARG, "device index out of range");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lk(g_mu);
    e = set_up(dev);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "set-up of the static scratch: %s", cudaGetErrorString(e));
        return err_arg(PKV_ERR_CUDA, msg);
    }
    unsigned char *base = static_cast<unsigned char *>(g_scratch_dev[dev]);

    // host image of the descriptor; pageable memory, staged by the driver
    // before cudaMemcpyAsync returns
    std::vector<unsigned char> blob(desc_end - rows_off, 0);
    std::memcpy(blob.data(), &row, sizeof row);
    if (!units.empty())
        std::memcpy(blob.data() + (units_off - rows_off), units.data(), units.size() * sizeof(UnitDesc));
    if (!tiles.empty())
        std::memcpy(blob.data() + (tiles_off - rows_off), tiles.data(), tiles.size() * sizeof(PrefillTile));
    if (!merges.empty())
        std::memcpy(blob.data() + (merges_off - rows_off), merges.data(), merges.size() * sizeof(MergeDesc));
    if (!items.empty()) {
        std::memcpy(blob.data() + (items_off - rows_off), items.data(), items.size() * sizeof(SplitItem));
        std::memcpy(blob.data() + (tile0_off - rows_off), img_tile0.data(), img_tile0.size() * sizeof(int32_t));
        std::memcpy(blob.data() + (slot_off - rows_off), img_slot.data(), img_slot.size() * sizeof(int32_t));
    }
    e = cudaMemcpyAsync(base + rows_off, blob.data(), blob.size(), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return err_arg(PKV_ERR_CUDA, cudaGetErrorString(e));

    AttnArgs a{};
    a.Q = Q;
    a.out = out;
    a.rows = reinterpret_cast<const RowDesc *>(base + rows_off);
    a.units = reinterpret_cast<const UnitDesc *>(base + units_off);
    a.merges = reinterpret_cast<const MergeDesc *>(base + merges_off);
    a.n_units = static_cast<int32_t>(units.size());
    a.n_heads = n_heads;
    a.n_kv = n_kv_heads;
    a.hd = head_dim;
    a.group = n_heads / n_kv_heads;
    a.causal = causal ? 1 : 0;
    a.split_keys = S;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.err = reinterpret_cast<int32_t *>(base);
    if (pf > 0) {
        a.pm = reinterpret_cast<float *>(base + part_off);
        a.pl = a.pm + pf;
        a.pacc = a.pl + pf;
    }
    const ContigAddr addr{Kc, Vc, n_kv_heads * head_dim};
    if (!tiles.empty()) {
        const SplitArgs sa{a.rows, reinterpret_cast<const SplitItem *>(base + items_off),
                           static_cast<int32_t>(items.size()), n_kv_heads, base + img_off, a.err};
        SplitCtx sc{&sa, &addr, st};
        e = launch_counted(PKV_KERNEL_SPLIT, st, run_split, &sc);
        PrefillArgs pa{Q, out, a.rows, reinterpret_cast<const PrefillTile *>(base + tiles_off),
                       static_cast<int32_t>(tiles.size()), a.pm, a.pl, a.pacc, n_heads,
                       n_kv_heads, a.group, a.causal, S * kPrefillSplitFactor, a.scale_log2,
                       a.err};
        pa.img = base + img_off;
        pa.img_tile0 = reinterpret_cast<const int32_t *>(base + tile0_off);
        pa.img_slot = reinterpret_cast<const int32_t *>(base + slot_off);
        PrefillCtx pc{&pa, &addr, st};
        if (e == cudaSuccess) e = launch_counted(PKV_KERNEL_PREFILL, st, run_prefill, &pc);
    }
    DecodeCtx dc{&a, &addr, st};
    if (e == cudaSuccess && !units.empty()) e = launch_counted(PKV_KERNEL_DECODE, st, run_decode, &dc);
    if (e == cudaSuccess && !merges.empty()) {
        MergeArgs m{a.pm, a.pl, a.pacc, out, a.rows,
                    reinterpret_cast<const MergeDesc *>(base + merges_off),
                    static_cast<int32_t>(merges.size()), n_heads, head_dim};
        MergeCtx mc{&m, st};
        e = launch_counted(PKV_KERNEL_MERGE, st, run_merge, &mc);
    }
    if (e != cudaSuccess) return err_arg(PKV_ERR_CUDA, cudaGetErrorString(e));
    return PKV_OK;
}
