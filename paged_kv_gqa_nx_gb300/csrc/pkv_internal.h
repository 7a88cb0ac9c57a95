// pkv_internal.h -- descriptors and kernel launchers shared by the host core
// (pkv_host.cpp) and the kernels (pkv_kernels.cu).  Not part of the C ABI.
#pragma once

#include <atomic>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

namespace pkv {

// One batch row: a sequence appending and attending n_q consecutive rows.
struct RowDesc {
    int32_t slot;      // page-table row of the sequence on the device
    int32_t past_len;  // tokens committed before this call (seq_len)
    int32_t n_q;       // rows appended and attended by this call
    int32_t q_row0;    // first of this row's rows in Q / K_new / V_new / out
    // Shared-prefix (cascade) rows: keys [0, k0) were attended by a prefix
    // pass whose partials are the first s0 records of the query's merge item;
    // the row's decode unit of split s covers k0 + (s - s0) * S .. (S keys).
    // 0, 0 for every other row.
    int32_t k0 = 0, s0 = 0;
};

// One split-K work unit: query qi of row `row`, keys [split*S, (split+1)*S)
// clipped to the visible range.  item >= 0: the query has several splits and
// MergeDesc `item` describes them (this unit's partial record is
// part0 + split); item < 0: the unit writes out directly.
struct UnitDesc {
    int32_t row, qi, split, item;
};

// One query whose splits are combined by the merge kernel.
struct MergeDesc {
    int32_t row, qi, part0, n_split;
};

// One appended token row: position `pos` (in block `blk` of the host page
// table) receives row `src_row` of K_new / V_new.
struct AppendDesc {
    int32_t slot, pos, src_row, blk;
};

// A run of page-table entries to upload: pt[slot][start .. start+count) =
// vals[voff .. voff+count).
struct PtRun {
    int32_t slot, start, count, voff;
};

// One copy-on-append block copy (every layer, K and V).
struct CopyDesc {
    int32_t src, dst;
};

// Address of a key/value row in the paged pool:
//   pool[pt[slot][pos / bs]][layer][pos % bs][kv_head*hd ...]
struct PagedAddr {
    void *k, *v;           // pool storage: f32 elements, or bf16 when bf16 != 0
    int32_t *pt;           // written only by the fused append, for pages no reader of that launch uses
    int64_t block_stride;  // elements per block: n_layers * bs * kv_dim
    int64_t layer_off;     // elements to the layer: layer * bs * kv_dim
    int32_t kv_dim, bs, bs_shift, max_blocks, n_blocks;
    int32_t bf16 = 0;      // storage element: 0 f32, 1 bf16 (rounded to nearest even on write)
    int32_t fp8 = 0;       // 1: fp8 e4m3 elements holding x / kv_scale (saturating)
    float kv_scale = 1.f;  // power of two; 1 unless fp8
};

// Address of a key/value row in a contiguous history: base[pos][kv_head*hd ...]
struct ContigAddr {
    const float *k, *v;
    int32_t kv_dim;
};

struct AttnArgs {
    const float *Q;
    float *out;
    const RowDesc *rows;
    const UnitDesc *units;
    const MergeDesc *merges;  // merge items of the units with several splits
    int32_t n_units;
    float *pm, *pl, *pacc;  // partials: [n_part][n_heads], [n_part][n_heads], [n_part][n_heads][hd]
    int32_t n_heads, n_kv, hd, group, causal, split_keys;
    float scale_log2;       // scale * log2(e): scores are kept in base-2 units
    int32_t *err;
    // Fused append (paged decode, K_new != nullptr): a row's positions
    // past_len .. past_len + n_q - 1 are read from K_new / V_new row
    // q_row0 + (pos - past_len) instead of the pool, and the unit of query
    // n_q - 1 whose split holds them also stores them into the pool (block id
    // app[q_row0 + t].blk) and, when pt_write is set, enters each new block
    // (a position at a block boundary) into the device page table.
    const float *K_new = nullptr, *V_new = nullptr;
    const AppendDesc *app = nullptr;
    int32_t pt_write = 0;
};

// One tensor-core prefill tile: queries q0 .. q0 + 128/G - 1 of row `row`
// (clipped to n_q), key split `split` of size PrefillArgs::split_keys.
// part0 < 0: the tile's queries have one split and write out directly;
// otherwise query q0 + t's partial for split s is record
// part0 + t*stride + s, stride = n_split unless the tile sets it (a prefix
// pass leaves room for the decode splits that follow each query's prefix).
// The kernel takes tiles in pairs, one pair per CTA: tiles 2i and 2i + 1 share
// the row and the split; row < 0 marks an absent second tile.
struct PrefillTile {
    int32_t row, q0, split, part0;
    int32_t stride = 0;
};

struct PrefillArgs {
    const float *Q;
    float *out;
    const RowDesc *rows;
    const PrefillTile *tiles;
    int32_t n_tiles;  // even: two per CTA
    float *pm, *pl, *pacc;  // same partial layout as AttnArgs
    int32_t n_heads, n_kv, group, causal, split_keys;
    float scale_log2;
    int32_t *err;
    // Paged launches: the K/V operand images made by the split pass (or kept
    // from earlier calls); row r's key tile kt for kv head h is image
    // img_slot[img_tile0[r] + kt] * n_kv + h.
    const unsigned char *img = nullptr;
    const int32_t *img_tile0 = nullptr;
    const int32_t *img_slot = nullptr;
    // the images' piece-1 planes are left out (a bf16 or fp8 pool: every K/V
    // value times the tile's power of two is an f16 value), so the products
    // with them and their copies are skipped
    int32_t lo_zero = 0;
};

// The tensor-core kernel's operands for one (row, 64-key tile, kv head), as
// they sit in its shared memory: K0, K1 (K-major, 128-byte swizzle, two
// k-blocks of 64 dims x 64 keys) and V0^T, V1^T (one k-block of 64 keys x
// 128 dims), f16; then the tile's two exponents (int32 K, V).  Each f32
// value x of the tile is x * 2^e = x0 + x1, x0 = f16(x * 2^e), x1 = f16 of the
// exact rest, e the tile's exponent (its largest magnitude into [2^14, 2^15)).
constexpr int32_t kKeyTile = 64;  // keys per tensor-core tile (and per image)
constexpr uint32_t kImagePlane = 16 * 1024;
constexpr uint32_t kImageExpOff = 4 * kImagePlane;
constexpr uint32_t kImageBytes = 4 * kImagePlane + 128;  // a multiple of 128 bytes

// One image to make: key tile kt of row `row` (all kv heads), into image
// slot `slot` (images slot * n_kv + h).
struct SplitItem {
    int32_t row, kt, slot;
};

struct SplitArgs {
    const RowDesc *rows;
    const SplitItem *items;
    int32_t n_items, n_kv;
    unsigned char *img;
    int32_t *err;
};

struct MergeArgs {
    const float *pm, *pl, *pacc;
    float *out;
    const RowDesc *rows;
    const MergeDesc *items;
    int32_t n_items, n_heads, hd;
};

// One launch before attention: upload page-table runs, append the new rows.
struct PrepArgs {
    int32_t *pt;
    int32_t max_blocks;
    const PtRun *runs;
    const int32_t *vals;
    int32_t n_runs;
    const AppendDesc *app;
    int32_t n_app;
    const float *K_new, *V_new;
    bool vec4;
    int32_t *err;
    // RoPE on append (rope_base > 0): K rows are rotated on their way into
    // the pool and Q rows into Q_rot, at position AppendDesc::pos; pairs
    // (i, i + hd/2) turn by pos * rope_base^(-2i/hd).
    double rope_base = 0.0;
    const float *Q = nullptr;
    float *Q_rot = nullptr;
    int32_t q_dim = 0, hd = 0;
};

// Set-up done once per device: a kernel's function attributes (its dynamic
// shared-memory opt-in) belong to the current device's context, so a process
// that drives several GPUs sets them on each.  Setting an attribute is
// idempotent, so threads that race here all set the same value.
struct PerDeviceOnce {
    std::atomic<uint64_t> done{0};  // bit d: device d is set up
    template <class F>
    cudaError_t run(F &&f) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
        if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
        e = f();
        if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
        return e;
    }
};

// Kernel launchers (pkv_kernels.cu).  Each enqueues exactly one kernel.
cudaError_t launch_prep(const PrepArgs &a, const PagedAddr &addr, cudaStream_t s);
cudaError_t launch_pt_apply(int32_t *pt_dev, int32_t max_blocks, const PtRun *runs, int32_t n_runs,
                            const int32_t *vals, cudaStream_t s);
// block_words: one block's K (or V) storage in 4-byte words
cudaError_t launch_copy_blocks(void *k, void *v, const CopyDesc *items, int32_t n_items,
                               int64_t block_words, int32_t n_blocks, int32_t *err,
                               cudaStream_t s);
cudaError_t launch_decode_paged(const AttnArgs &a, const PagedAddr &addr, cudaStream_t s);
cudaError_t launch_decode_contig(const AttnArgs &a, const ContigAddr &addr, cudaStream_t s);
// Decode over a bf16 or fp8 pool on the tensor cores (pkv_decode_mma.cu), for
// the shapes decode_mma_shape accepts; with AttnArgs::K_new it also takes the
// fused append (the new rows rounded to the pool element as the append does).
cudaError_t launch_decode_mma_paged(const AttnArgs &a, const PagedAddr &addr, cudaStream_t s);
__host__ __device__ constexpr bool decode_mma_shape(int head_dim, int group, bool bf16, bool fp8) {
    return head_dim == 128 &&
           ((fp8 && (group == 1 || group == 2 || group == 4 || group == 8)) ||
            (!fp8 && bf16 && (group == 1 || group == 2 || group == 4)));
}
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s);
// Tensor-core prefill (pkv_prefill.cu): head_dim 128, group 1, 2, 4 or 8; its
// K/V operands are the images in PrefillArgs::img (made by the split pass).
cudaError_t launch_prefill_paged(const PrefillArgs &a, const PagedAddr &addr, cudaStream_t s);
cudaError_t launch_prefill_contig(const PrefillArgs &a, const ContigAddr &addr, cudaStream_t s);
// The split pass of the tensor-core launches: one image per item and kv head,
// from the pool's rows or from a contiguous K/V pair.
cudaError_t launch_split_paged(const SplitArgs &a, const PagedAddr &addr, cudaStream_t s);
cudaError_t launch_split_contig(const SplitArgs &a, const ContigAddr &addr, cudaStream_t s);

// Rows with at least this many queries take the tensor-core prefill kernel
// (when head_dim is 128 and the group is 1, 2, 4 or 8); its key split is
// kPrefillSplitFactor times the decode split.  Both depend only on the row.
constexpr int kPrefillMinQueries = 32;
constexpr int kPrefillSplitFactor = 16;
__host__ __device__ constexpr bool prefill_shape(int head_dim, int group) {
    return head_dim == 128 && (group == 1 || group == 2 || group == 4 || group == 8);
}

// Host-core helpers for entry points defined in other translation units
// (pkv_host.cpp).  build_contig_work: the split-K work list of one contiguous
// row, as pkv_attn_contiguous builds it (allow_tc false: no tensor-core
// tiles, every query to the split-K decode kernels).  launch_counted: enqueue fn(ctx) with
// the library's launch accounting and optional event timing.  report_error:
// record the calling thread's last error message and return code.
void build_contig_work(int32_t n_q, int32_t total_k, int32_t causal, int32_t split_keys,
                       int32_t head_dim, int32_t group, std::vector<UnitDesc> &units,
                       std::vector<PrefillTile> &tiles, std::vector<MergeDesc> &merges,
                       int64_t *n_part, bool allow_tc = true);
cudaError_t launch_counted(int kind, cudaStream_t s, cudaError_t (*fn)(void *), void *ctx);
int32_t current_split_keys();
int report_error(int code, const char *msg);
// The error word of pkv_attn_contiguous_noalloc on device `dev` (current): its
// device address, or nullptr when no call has set it up yet and `setup` is
// false; with `setup`, the first use on the device sets it up (*e reports a
// failure).  Defined in pkv_noalloc.cu.
int32_t *noalloc_error_word(int dev, bool setup, cudaError_t *e);

// Largest head_dim the decode kernels accept.
constexpr int kMaxHeadDim = 256;

}  // namespace pkv
