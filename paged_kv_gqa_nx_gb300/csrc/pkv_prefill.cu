// pkv_prefill.cu -- tensor-core attention for chunked-prefill rows (n_q > 1).
//
// For a row with many new tokens, Q.K^T over a tile of queries and keys is a
// real dense contraction, so it runs on the 5th-generation tensor cores
// (tcgen05.mma kind::tf32).  To keep f32 accuracy each f32 operand x is split
// into a tf32 part and its exact f32 rest (x = hi + lo) and every product is
// formed as hi*hi + hi*lo + lo*hi; the dropped lo*lo term is ~2^-20 relative.
//
// One CTA = one tile of 128 query rows -- (128 / G) consecutive tokens x the G
// query heads that share kv head `kvh` -- and one key split.  16 compute
// warps and one more warpgroup whose first warp issues the MMAs; that
// warpgroup hands most of its registers to the compute warps (setmaxnreg),
// which keeps the compute warps' prefetch registers from spilling.  Row m of
// the tile is token m / G, head m % G
// and TMEM lane m; the four compute threads that share TMEM lane m (warps w,
// w + 4, w + 8, w + 12) each own 16 of a key tile's scores and 32 of the row's
// output columns, and combine the row max and sum through shared memory.  The
// compute warps arrive on an mbarrier when the operands of QK or PV are in
// place; the issue warp waits on it, issues, and commits to the mbarrier the
// compute warps wait on.  Key tiles are 64 positions:
//   QK(j):  S[128 x 64]  = Q.K_j^T     A = Q hi (TMEM) / Q lo (smem), B = K_j (smem)
//   PV(j):  D[128 x 128] = P_j.V_j     A = P hi/lo (TMEM),            B = V_j^T (smem)
// Loop j: wait S_j -> write K_{j+1} (QK(j+1) starts) -> online softmax
// (offset-causal mask: key p visible iff p <= q_pos = total_k - n_q + i) ->
// wait PV(j-1) -> write P_j, V_j (PV(j) starts, adding into the TMEM
// accumulator D); QK(j+1) runs during the softmax of tile j.  p is
// relative to a reference max that moves (and D is rescaled) only when a
// tile's max exceeds it by more than 2^8, which keeps every p below 256.
// K/V rows for the next tiles are loaded into registers while the MMAs run.
// Shared memory: Q lo 64 KiB, K hi/lo 64 KiB, V^T hi/lo 64 KiB.
// TMEM (512 columns): Q hi [0,128), S [128,192), P hi [256,320), P lo
// [320,384), D [384,512).
//
// The address functors mirror the decode kernels' (paged through the page
// table, or contiguous), so the paged and contiguous instantiations return the
// same bits.
#include "pkv_elem.h"
#include "pkv_internal.h"
#include "pkv_tcgen05.h"

#include <type_traits>

namespace pkv {
namespace {

using namespace tc;

constexpr int kHD = 128;
constexpr int kKT = 64;  // keys per tile
static_assert(kKT == kKeyTile, "one image per tile");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQhi = 0, kColS = 128, kColPhi = 256, kColPlo = 320, kColD = 384;
#ifndef PKV_PREFILL_COMPUTE_WARPS
#define PKV_PREFILL_COMPUTE_WARPS 16
#endif
constexpr int kComputeWarps = PKV_PREFILL_COMPUTE_WARPS;  // 8: two threads per tile row, 16: four
constexpr int kCompute = 32 * kComputeWarps;
// + one warpgroup whose first warp issues the MMAs; it gives registers back
// (setmaxnreg) so that the compute warps can hold more
constexpr int kThreads = kCompute + 128;
// per thread at launch: 65536 registers over the CTA, and 16384 over the at
// most kThreads/128 warps of one SM sub-partition
constexpr int kLaunchRegs = kComputeWarps == 16 ? 96 : 168;
constexpr int kIssueRegs = 32;                                 // issue warpgroup after .dec
constexpr int kComputeRegs = kComputeWarps == 16 ? 112 : 232;  // compute warps after .inc
static_assert(kCompute * kComputeRegs + 128 * kIssueRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch's registers");
// with operand images the compute warps hold no prefetch registers and the
// issue thread also runs the copies
constexpr int kIssueRegsBulk = 80;
constexpr int kComputeRegsBulk = kComputeWarps == 16 ? 96 : 184;
static_assert(kCompute * kComputeRegsBulk + 128 * kIssueRegsBulk <= kThreads * kLaunchRegs,
              "register split exceeds the launch's registers");
static_assert(kComputeWarps != 16 || 4 * 32 * kComputeRegsBulk + 32 * kIssueRegsBulk <= 16384,
              "register split exceeds one SM sub-partition");
constexpr int kTPR = kComputeWarps / 4;                     // threads per tile row
constexpr int kSCols = kKT / kTPR;                          // scores per thread per key tile
constexpr int kDCols = kHD / kTPR;                          // output columns per thread
constexpr int kKPW = kKT / kComputeWarps;                   // K rows per warp per key tile
static_assert(kComputeWarps == 8 || kComputeWarps == 16, "8 or 16 compute warps");
constexpr float kRescale = 8.f;               // lazy-rescale threshold (base 2)

template <class E>
struct PagedRowsP {
    using Elem = E;
    PagedAddr a;
    // Block id of (slot, pos), or -1 (and the error flag) when the page index
    // or the id is out of range.
    __device__ __forceinline__ int block(int slot, int pos, int32_t *err) const {
        const int bi = a.bs_shift >= 0 ? (pos >> a.bs_shift) : (pos / a.bs);
        if (bi >= a.max_blocks) {
            if (err) atomicOr(err, 1);
            return -1;
        }
        const int blk = __ldg(a.pt + static_cast<size_t>(slot) * a.max_blocks + bi);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.n_blocks)) {
            if (err) atomicOr(err, 1);
            return -1;
        }
        return blk;
    }
    // The page-table entry of (slot, pos) without waiting for it: -1 when the
    // page index is out of range (error flag set), else the raw entry, which
    // checked() validates where it is used, a tile later, so the lookup's
    // latency stays off the critical path.
    __device__ __forceinline__ int entry(int slot, int pos, int32_t *err) const {
        const int bi = a.bs_shift >= 0 ? (pos >> a.bs_shift) : (pos / a.bs);
        if (bi >= a.max_blocks) {
            if (err) atomicOr(err, 1);
            return -1;
        }
        return __ldg(a.pt + static_cast<size_t>(slot) * a.max_blocks + bi);
    }
    __device__ __forceinline__ int checked(int blk, int32_t *err) const {
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.n_blocks)) {
            if (err) atomicOr(err, 1);
            return -1;
        }
        return blk;
    }
    __device__ __forceinline__ size_t offset(int blk, int pos, int kvh) const {
        const int off = a.bs_shift >= 0 ? (pos & (a.bs - 1)) : (pos % a.bs);
        return static_cast<size_t>(blk) * a.block_stride + a.layer_off +
               static_cast<size_t>(off) * a.kv_dim + static_cast<size_t>(kvh) * kHD;
    }
    __device__ __forceinline__ const E *k_row(int blk, int pos, int kvh) const {
        return static_cast<const E *>(a.k) + offset(blk, pos, kvh);
    }
    __device__ __forceinline__ const E *v_row(int blk, int pos, int kvh) const {
        return static_cast<const E *>(a.v) + offset(blk, pos, kvh);
    }
    // groups of n positions starting at a multiple of n lie in one block
    __device__ __forceinline__ bool whole(int n) const { return (a.bs % n) == 0; }
};

struct ContigRowsP {
    using Elem = float;
    ContigAddr a;
    __device__ __forceinline__ int block(int, int, int32_t *) const { return 0; }
    __device__ __forceinline__ int entry(int, int, int32_t *) const { return 0; }
    __device__ __forceinline__ int checked(int blk, int32_t *) const { return blk; }
    __device__ __forceinline__ const float *k_row(int, int pos, int kvh) const {
        return a.k + static_cast<size_t>(pos) * a.kv_dim + static_cast<size_t>(kvh) * kHD;
    }
    __device__ __forceinline__ const float *v_row(int, int pos, int kvh) const {
        return a.v + static_cast<size_t>(pos) * a.kv_dim + static_cast<size_t>(kvh) * kHD;
    }
    __device__ __forceinline__ bool whole(int) const { return true; }
};

constexpr uint32_t kSmemQlo = 64 * 1024;  // 4 k-blocks of 128 rows
constexpr uint32_t kSmemK = 32 * 1024;    // one of K hi / lo: 4 k-blocks of 64 rows
constexpr uint32_t kSmemV = 32 * 1024;    // one of V^T hi / lo: 2 k-blocks of 128 rows
constexpr size_t kSmemBytes = kSmemQlo + 2 * kSmemK + 2 * kSmemV + 1024;  // + alignment slack

__device__ __forceinline__ void split4(const float4 &x, float4 &h, float4 &l) {
    split_tf32(x.x, h.x, l.x);
    split_tf32(x.y, h.y, l.y);
    split_tf32(x.z, h.z, l.z);
    split_tf32(x.w, h.w, l.w);
}

// kBulk: the K/V operands come as images (the split pass) by bulk copy;
// otherwise the compute warps load and split them.  kLoZero (images of a bf16
// pool): the K / V lo planes are zero, so they are neither copied nor used.
template <int G, class Rows, bool kBulk, bool kLoZero>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(PrefillArgs a, Rows rows_of) {
    constexpr int TQ = 128 / G;  // tokens per tile
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *Qlo = sm;
    unsigned char *Khi = Qlo + kSmemQlo;
    unsigned char *Klo = Khi + kSmemK;
    unsigned char *Vhi = Klo + kSmemK;
    unsigned char *Vlo = Vhi + kSmemV;
    // bar_qk / bar_pv: the MMAs of QK / PV completed (tcgen05.commit);
    // bar_k / bar_p: the operands of QK / PV are in place.  Register mode: the
    // compute warps stored them.  Image mode: the compute warps read S (or, the
    // first time, wrote Q) / wrote P, and the copy warp's K / V image landed.
    __shared__ uint64_t bar_qk, bar_pv, bar_k, bar_p;
    __shared__ uint32_t tslot;
    __shared__ float red[2][kCompute];
    static_assert(kSCols == 16 || kSCols == 32, "");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ti = blockIdx.x / a.n_kv;
    const int kvh = blockIdx.x - ti * a.n_kv;
    const PrefillTile tile = a.tiles[ti];
    const RowDesc rd = a.rows[tile.row];
    const int total_k = rd.past_len + rd.n_q;
    const int n_valid_q = min(TQ, rd.n_q - tile.q0);
    const int kend_tile =
        a.causal ? min(total_k, total_k - rd.n_q + tile.q0 + n_valid_q) : total_k;
    const int kbeg = tile.split * a.split_keys;
    const int kend = min(kbeg + a.split_keys, kend_tile);
    const int kt0 = kbeg / kKT, kt1 = (kend + kKT - 1) / kKT;

    if (warp == 0) {
        tmem_alloc(smem_u32(&tslot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_u32(&bar_qk), 1);
        mbar_init(smem_u32(&bar_pv), 1);
        // with images the copy warp's expect-tx arrival joins each phase
        mbar_init(smem_u32(&bar_k), kComputeWarps + (kBulk ? 1 : 0));
        mbar_init(smem_u32(&bar_p), kComputeWarps + (kBulk ? 1 : 0));
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;
    bool ok = true;

    if (warp >= kComputeWarps) {
        // the issue warpgroup: its first warp issues the MMAs, in image mode
        // its second warp runs the bulk copies; the rest only give their
        // registers back
        setmaxnreg_dec<kBulk ? kIssueRegsBulk : kIssueRegs>();
        if (kBulk && warp == kComputeWarps + 1) {
            // ---------------- copy warp (lane 0 copies) ----------------
            // A K / V buffer is refilled as soon as the MMAs that read it are
            // done, in the order the tensor core completes them: QK(kt0), then
            // QK(kt+1), PV(kt), ...  Each copy arrives with its byte count on
            // the operand barrier that the MMA warp waits on.
            // tile kt's image slot; read a copy ahead of its use (slot_at is
            // called only by lane 0)
            const int32_t *slots = a.img_slot + a.img_tile0[tile.row];
            auto slot_at = [&](int kt) { return kt < kt1 ? __ldg(slots + kt) : 0; };
            auto image = [&](int32_t slot) {
                return a.img + (static_cast<size_t>(slot) * a.n_kv + kvh) * kImageBytes;
            };
            constexpr uint32_t planes = kLoZero ? 1u : 2u;  // hi (and lo) of K / V
            auto copy_k = [&](int32_t slot) {
                if (lane == 0) {
                    const unsigned char *src = image(slot);
                    mbar_expect_tx(smem_u32(&bar_k), planes * kImagePlane);
                    bulk_g2s(smem_u32(Khi), src, kImagePlane, smem_u32(&bar_k));
                    if constexpr (planes == 2) bulk_g2s(smem_u32(Klo), src + kImagePlane, kImagePlane, smem_u32(&bar_k));
                }
            };
            auto copy_v = [&](int32_t slot) {
                if (lane == 0) {
                    const unsigned char *src = image(slot) + 2 * kImagePlane;
                    mbar_expect_tx(smem_u32(&bar_p), planes * kImagePlane);
                    bulk_g2s(smem_u32(Vhi), src, kImagePlane, smem_u32(&bar_p));
                    if constexpr (planes == 2) bulk_g2s(smem_u32(Vlo), src + kImagePlane, kImagePlane, smem_u32(&bar_p));
                }
            };
            auto wait_c = [&](uint64_t *bar, uint32_t &ph) {
                const bool w = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(smem_u32(bar), ph) : true, 0);
                ph ^= 1;
                return w;
            };
            uint32_t ph_qkd = 0, ph_pvd = 0;
            bool cok = true;
            int32_t s_v = 0, s_k = 0;  // slots of the next V copy (kt + 1) and K copy (kt + 2)
            if (lane == 0 && kt0 < kt1) {
                const int32_t s0 = slot_at(kt0);
                s_v = slot_at(kt0 + 1);
                s_k = slot_at(kt0 + 2);
                copy_k(s0);
                copy_v(s0);
            }
            if (kt0 + 1 < kt1) {
                cok = wait_c(&bar_qk, ph_qkd);  // QK(kt0) done
                if (cok) copy_k(s_v);
            }
            for (int kt = kt0; kt + 1 < kt1 && cok; ++kt) {
                if (kt + 2 < kt1) {
                    cok = wait_c(&bar_qk, ph_qkd);  // QK(kt+1) done: the K buffer is free
                    if (!cok) break;
                    copy_k(s_k);
                }
                cok = wait_c(&bar_pv, ph_pvd);  // PV(kt) done: the V buffer is free
                if (!cok) break;
                copy_v(s_v);
                if (lane == 0) {
                    s_v = s_k;
                    s_k = slot_at(kt + 3);
                }
            }
            // let the last copies land before the CTA's shared memory is given
            // up (their phases also need the compute warps; bounded if those
            // gave up)
            if (kt0 < kt1) {
                uint32_t last = static_cast<uint32_t>(kt1 - 1 - kt0) & 1u;
                wait_c(&bar_k, last);
                last = static_cast<uint32_t>(kt1 - 1 - kt0) & 1u;
                wait_c(&bar_p, last);
            }
        } else if (warp == kComputeWarps) {
        // ---------------- MMA issue warp (lane 0 issues) ----------------
        const uint64_t dKhi = desc_sw128(smem_u32(Khi)), dKlo = desc_sw128(smem_u32(Klo));
        const uint64_t dQlo = desc_sw128(smem_u32(Qlo));
        const uint64_t dVhi = desc_sw128(smem_u32(Vhi)), dVlo = desc_sw128(smem_u32(Vlo));
        const uint32_t tS = tbase + kColS, tQ = tbase + kColQhi, tD = tbase + kColD;
        const uint32_t tPh = tbase + kColPhi, tPl = tbase + kColPlo;
        const uint32_t idesc_s = idesc_tf32(128, kKT), idesc_o = idesc_tf32(128, kHD);
        uint32_t ph_k = 0, ph_p = 0;
        // one k-step of QK (8 dims) / PV (8 keys): three products of the split
        // (products with the K / V lo planes are left out when those are zero)
        constexpr bool lo = !kLoZero;
        auto qk_step = [&](int s) {
            const uint64_t ko = ((s >> 2) * 8192u + (s & 3) * 32u) >> 4;
            const uint64_t qo = ((s >> 2) * 16384u + (s & 3) * 32u) >> 4;
            mma_tf32_ts(tS, tQ + 8 * s, dKhi + ko, idesc_s, s > 0);
            if constexpr (lo) mma_tf32_ts(tS, tQ + 8 * s, dKlo + ko, idesc_s, 1);
            mma_tf32(tS, dQlo + qo, dKhi + ko, idesc_s, 1);
        };
        auto pv_step = [&](int s, bool first) {
            const uint64_t vo = ((s >> 2) * 16384u + (s & 3) * 32u) >> 4;
            mma_tf32_ts(tD, tPh + 8 * s, dVhi + vo, idesc_o, !first || s > 0);
            if constexpr (lo) mma_tf32_ts(tD, tPh + 8 * s, dVlo + vo, idesc_o, 1);
            mma_tf32_ts(tD, tPl + 8 * s, dVhi + vo, idesc_o, 1);
        };
        // the MMAs of one tile (lane 0 issues, then commits); unrolled when the
        // issue warpgroup has the registers for it (image mode)
        auto mma_qk = [&]() {
            fence_after_sync();
            if (lane == 0) {
                if constexpr (kBulk) {
#pragma unroll
                    for (int s = 0; s < 16; ++s) qk_step(s);
                } else {
#pragma unroll 1
                    for (int s = 0; s < 16; ++s) qk_step(s);
                }
                mma_commit(smem_u32(&bar_qk));
            }
            __syncwarp();
        };
        auto mma_pv = [&](bool first) {
            fence_after_sync();
            if (lane == 0) {
                if constexpr (kBulk) {
#pragma unroll
                    for (int s = 0; s < 8; ++s) pv_step(s, first);
                } else {
#pragma unroll 1
                    for (int s = 0; s < 8; ++s) pv_step(s, first);
                }
                mma_commit(smem_u32(&bar_pv));
            }
            __syncwarp();
        };
        // lane 0 waits (bounded), the warp learns the outcome
        auto wait1 = [&](uint64_t *bar, uint32_t &ph) {
            const bool w = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(smem_u32(bar), ph) : true, 0);
            ph ^= 1;
            return w;
        };
        // order on the tensor core: QK(kt0), then per tile QK(kt+1) before
        // PV(kt), so QK(kt+1) runs while the compute warps do the softmax
        if (kt0 < kt1) {
            ok = wait1(&bar_k, ph_k);  // K of the tile (and, the first time, Q) in place
            if (ok) mma_qk();
        }
        for (int kt = kt0; kt < kt1 && ok; ++kt) {
            if (kt + 1 < kt1) {
                ok = wait1(&bar_k, ph_k);
                if (!ok) break;
                mma_qk();
            }
            ok = wait1(&bar_p, ph_p);  // P and V of the tile in place
            if (!ok) break;
            mma_pv(kt == kt0);
        }
        if (!ok && lane == 0 && a.err) atomicOr(a.err, 2);
        }
    } else {
        setmaxnreg_inc<kBulk ? kComputeRegsBulk : kComputeRegs>();
        // ---------------- compute warps: 4 threads per tile row ----------------
        const int wq = warp & 3;               // TMEM lane quadrant
        const int qp = warp >> 2;              // which quarter of the row this thread owns
        const int m = 32 * wq + lane;          // this thread's row of the tile
        const int tq = m / G, g = m - (m / G) * G;
        const int qi = tile.q0 + tq;
        const bool valid = qi < rd.n_q;
        const int q_pos = total_k - rd.n_q + qi;
        const int kend_row = valid ? (a.causal ? min(q_pos + 1, total_k) : total_k) : 1;
        const uint32_t tlane = static_cast<uint32_t>(32 * wq) << 16;

        // Q row (pre-scaled to base-2 units): this thread's kDCols dims, hi -> TMEM,
        // lo -> shared memory (one k-block per 32 dims)
        {
            const float *qrow = a.Q + static_cast<size_t>(rd.q_row0 + (valid ? qi : 0)) * (a.n_heads * kHD) +
                                static_cast<size_t>(kvh * G + g) * kHD + kDCols * qp;
#pragma unroll
            for (int c = 0; c < kDCols / 32; ++c) {
                float hv[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (valid) x = __ldg(reinterpret_cast<const float4 *>(qrow + 32 * c) + j4);
                    x.x *= a.scale_log2;
                    x.y *= a.scale_log2;
                    x.z *= a.scale_log2;
                    x.w *= a.scale_log2;
                    float4 h, l;
                    split4(x, h, l);
                    hv[4 * j4] = h.x;
                    hv[4 * j4 + 1] = h.y;
                    hv[4 * j4 + 2] = h.z;
                    hv[4 * j4 + 3] = h.w;
                    const uint32_t kb = static_cast<uint32_t>(kDCols / 32 * qp + c);
                    *reinterpret_cast<float4 *>(Qlo + kb * 16384u + sw128_chunk(m, j4)) = l;
                }
                tmem_st32(tbase + tlane + kColQhi + kDCols * qp + 32 * c, hv);
            }
        }

        // Key rows of a tile: warp w owns keys kKPW*w .. kKPW*w + kKPW-1 of both K
        // and V, so one page-table lookup per warp serves a tile when a block
        // holds whole kKPW-key groups.  K: one 512-byte row per instruction,
        // stored as 16-byte chunks of the K-major layout.  V: lane l loads dims
        // l + 32c (c < 4) of each row (128-byte coalesced loads) and writes
        // 16-byte runs of 4 keys into rows d = l + 32c of V^T; the 32 rows of one
        // store fall in all 8 swizzle phases, so the store is conflict-free.
        // Page-table lookups are issued one phase before the loads that use them.
        float4 kreg[kKPW], vq[kKPW / 4][4];
        const bool k_whole = rows_of.whole(kKPW);
        auto k_pos = [&](int kt) { return kt * kKT + warp * kKPW; };
        // row pointer of key pos (nullptr beyond the split or on a bad entry)
        using E = typename Rows::Elem;
        auto row_of = [&](int pos, int blk0, bool is_v) -> const E * {
            if (pos >= kend) return nullptr;
            int b = blk0;
            if (!k_whole) b = rows_of.block(rd.slot, pos, a.err);
            if (b < 0) return nullptr;
            return is_v ? rows_of.v_row(b, pos, kvh) : rows_of.k_row(b, pos, kvh);
        };
        auto load_k = [&](int kt, int blk0) {
            const int pos0 = k_pos(kt);
            if (k_whole && pos0 < kend) blk0 = rows_of.checked(blk0, a.err);
#pragma unroll
            for (int i = 0; i < kKPW; ++i) {
                const E *kr = row_of(pos0 + i, blk0, false);
                kreg[i] = kr ? ldg4(kr + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        auto load_v = [&](int kt, int blk0) {
            const int pos0 = k_pos(kt);
            if (k_whole && pos0 < kend) blk0 = rows_of.checked(blk0, a.err);
#pragma unroll
            for (int g4 = 0; g4 < kKPW / 4; ++g4) {
                float v[4][4];  // [key][c]
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const E *vr = row_of(pos0 + 4 * g4 + i, blk0, true);
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[i][c] = vr ? ldg1(vr + lane + 32 * c) : 0.f;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) vq[g4][c] = make_float4(v[0][c], v[1][c], v[2][c], v[3][c]);
            }
        };
        auto lookup_k = [&](int kt) {
            const int pos0 = k_pos(kt);
            return (k_whole && pos0 < kend) ? rows_of.entry(rd.slot, pos0, a.err) : -1;
        };
        auto lookup_v = lookup_k;
        auto store_k = [&]() {
#pragma unroll
            for (int i = 0; i < kKPW; ++i) {
                float4 h, l;
                split4(kreg[i], h, l);
                const uint32_t off = (lane >> 3) * 8192u + sw128_chunk(warp * kKPW + i, lane & 7);
                *reinterpret_cast<float4 *>(Khi + off) = h;
                *reinterpret_cast<float4 *>(Klo + off) = l;
            }
        };
        auto store_v = [&]() {
#pragma unroll
            for (int g4 = 0; g4 < kKPW / 4; ++g4) {
                const int key0 = warp * kKPW + 4 * g4;
                const uint32_t kb = static_cast<uint32_t>(key0 >> 5) * 16384u;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float4 h, l;
                    split4(vq[g4][c], h, l);
                    const uint32_t off = kb + sw128_chunk(lane + 32 * c, (key0 & 31) >> 2);
                    *reinterpret_cast<float4 *>(Vhi + off) = h;
                    *reinterpret_cast<float4 *>(Vlo + off) = l;
                }
            }
        };
        // Wait for an MMA commit: one thread polls the mbarrier and the others
        // wait in the named barrier, so the polling takes no shared-memory
        // bandwidth from the tensor core's operand reads.
        auto wait_one = [&](uint64_t *bar, uint32_t ph) {
            bool w = true;
            if (tid == 0) w = mbar_wait(smem_u32(bar), ph);
            __syncwarp();
            return named_sync_and(1, kCompute, w);
        };
        // operands written: make them visible to the tensor core, then one lane
        // per warp arrives on the barrier the issue warp waits on
        auto arrive = [&](uint64_t *bar) {
            tmem_st_wait();
            fence_proxy_async();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(bar));
        };

        // The output accumulator lives in TMEM (D) and the P.V MMAs add into it.
        // p is taken relative to a reference max m_ref that moves only when a
        // tile's max exceeds it by more than kRescale (base-2 units); then D and
        // l are rescaled once.  The four threads of a row take the same decisions.
        float m_ref = -INFINITY, l_run = 0.f;
        uint32_t ph_qk = 0, ph_pv = 0;

        // prologue: K_kt0 in place (QK(kt0) may start), V_kt0 and K_kt0+1 in
        // registers, the page-table entries of K_kt0+2 and V_kt0+1 on their way.
        // With images (kBulk) the issue thread brings K and V in: Q only.
        int vblk = -1, kblk = -1;
        if constexpr (!kBulk) {
            load_k(kt0, lookup_k(kt0));
            vblk = lookup_v(kt0);
            load_v(kt0, vblk);
            store_k();
            kblk = kt0 + 1 < kt1 ? lookup_k(kt0 + 1) : -1;
        }
        arrive(&bar_k);
        if constexpr (!kBulk) {
            if (kt0 + 1 < kt1) load_k(kt0 + 1, kblk);
            vblk = kt0 + 1 < kt1 ? lookup_v(kt0 + 1) : -1;
        }

        for (int kt = kt0; kt < kt1; ++kt) {
            // S_kt ready (QK(kt) done: the K buffer is free again)
            ok = wait_one(&bar_qk, ph_qk);
            ph_qk ^= 1;
            if (!ok) break;
            fence_after_sync();
            float s[kSCols];
            tmem_ldn<kSCols>(tbase + tlane + kColS + kSCols * qp, s);
            if constexpr (kBulk) {
                // S read: QK(kt+1) may overwrite it
                if (kt + 1 < kt1) arrive(&bar_k);
            } else if (kt + 1 < kt1) {
                // K_{kt+1} -> smem; the issue warp starts QK(kt+1) while we do
                // the softmax, and the K_{kt+2} loads overlap it too
                store_k();
                kblk = kt + 2 < kt1 ? lookup_k(kt + 2) : -1;
                arrive(&bar_k);
            }

            // online softmax: this thread's kSCols scores; max and sum combined over
            // the row's threads (tid + 128 k), in order of k
            const int base = kt * kKT + kSCols * qp;
            float tmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < kSCols; ++i) {
                const bool vis = base + i < kend_row && base + i < kend;
                s[i] = vis ? s[i] : -INFINITY;
                tmax = fmaxf(tmax, s[i]);
            }
            red[0][tid] = tmax;
            named_sync(1, kCompute);
            const int r0 = tid & 127;
            float row_max = red[0][r0];
#pragma unroll
            for (int k = 1; k < kTPR; ++k) row_max = fmaxf(row_max, red[0][r0 + 128 * k]);
            const bool rescale = m_ref != -INFINITY && row_max > m_ref + kRescale;
            const float m_use = (m_ref == -INFINITY || rescale) ? row_max : m_ref;
            float psum = 0.f;
#pragma unroll
            for (int i = 0; i < kSCols; ++i) {
                s[i] = (s[i] == -INFINITY) ? 0.f : exp2f(s[i] - m_use);
                psum += s[i];
            }
            red[1][tid] = psum;
            named_sync(1, kCompute);
            float rowsum = red[1][r0];
#pragma unroll
            for (int k = 1; k < kTPR; ++k) rowsum += red[1][r0 + 128 * k];

            // PV(kt-1) done: D, the P columns and the V buffer are free
            if (kt > kt0) {
                ok = wait_one(&bar_pv, ph_pv);
                ph_pv ^= 1;
                if (!ok) break;
                fence_after_sync();
            }
            // tcgen05.ld / st are warp-collective: the whole warp takes this branch
            // when any of its rows rescales (the others multiply by 1)
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? exp2f(m_ref - m_use) : 1.f;
#pragma unroll
                for (int c = 0; c < kDCols / 32; ++c) {
                    float dv[32];
                    tmem_ld32(tbase + tlane + kColD + kDCols * qp + 32 * c, dv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) dv[i] *= f;
                    tmem_st32(tbase + tlane + kColD + kDCols * qp + 32 * c, dv);
                    tmem_st_wait();
                }
                l_run *= f;
            }
            l_run += rowsum;
            m_ref = m_use;

            // P_kt -> TMEM (hi, then lo), V_kt -> smem; the issue warp starts PV(kt)
            {
                // hi from a copy, then lo in place (s is dead after this)
                float t[kSCols];
#pragma unroll
                for (int i = 0; i < kSCols; ++i) t[i] = __uint_as_float(__float_as_uint(s[i]) & 0xFFFFE000u);
                tmem_stn<kSCols>(tbase + tlane + kColPhi + kSCols * qp, t);
#pragma unroll
                for (int i = 0; i < kSCols; ++i) s[i] -= t[i];
                tmem_st_wait();
                tmem_stn<kSCols>(tbase + tlane + kColPlo + kSCols * qp, s);
            }
            if constexpr (!kBulk) store_v();
            arrive(&bar_p);

            // registers for the next tile: V_{kt+1}
            if constexpr (!kBulk) {
                if (kt + 1 < kt1) {
                    load_v(kt + 1, vblk);
                    vblk = kt + 2 < kt1 ? lookup_v(kt + 2) : -1;
                }
                if (kt + 2 < kt1) load_k(kt + 2, kblk);
            }
        }
        // the last PV, then the result
        if (ok) ok = wait_one(&bar_pv, ph_pv);
        if (!ok) {
            if (tid == 0 && a.err) atomicOr(a.err, 2);
        } else {
            fence_after_sync();
            const int h = kvh * G + g;
            const bool direct = tile.part0 < 0;
            float *dst = nullptr;
            size_t ph = 0;
            if (direct) {
                dst = a.out + static_cast<size_t>(rd.q_row0 + (valid ? qi : 0)) * (a.n_heads * kHD) +
                      static_cast<size_t>(h) * kHD + kDCols * qp;
            } else {
                const int n_split = (kend_tile + a.split_keys - 1) / a.split_keys;
                const int stride = tile.stride > 0 ? tile.stride : n_split;
                ph = static_cast<size_t>(tile.part0 + (valid ? tq : 0) * stride + tile.split) * a.n_heads + h;
                dst = a.pacc + ph * kHD + kDCols * qp;
            }
            const float scl = direct ? 1.f / l_run : 1.f;
#pragma unroll
            for (int c = 0; c < kDCols / 32; ++c) {
                float dv[32];
                tmem_ld32(tbase + tlane + kColD + kDCols * qp + 32 * c, dv);
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + 32 * c + i) =
                            make_float4(dv[i] * scl, dv[i + 1] * scl, dv[i + 2] * scl, dv[i + 3] * scl);
                }
            }
            if (valid) {
                if (!direct && qp == 0) {
                    a.pm[ph] = m_ref;
                    a.pl[ph] = l_run;
                }
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

template <int G, class Rows, bool kBulk, bool kLoZero>
cudaError_t launch_prefill_g(const PrefillArgs &a, const Rows &r, cudaStream_t s) {
    static PerDeviceOnce configured;  // the attribute is per function and device
    const cudaError_t ce = configured.run([&]() -> cudaError_t {
        // setmaxnreg.inc waits until the CTA's pool holds the registers it asks
        // for, so launch only if the compiled kernel starts with the registers
        // the split was sized for
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<G, Rows, kBulk, kLoZero>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < kLaunchRegs || fa.maxThreadsPerBlock < kThreads)
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(prefill_tc_kernel<G, Rows, kBulk, kLoZero>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        return cudaSuccess;
    });
    if (ce != cudaSuccess) return ce;
    const long long grid = static_cast<long long>(a.n_tiles) * a.n_kv;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prefill_tc_kernel<G, Rows, kBulk, kLoZero><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, s>>>(a, r);
    return cudaGetLastError();
}

template <class Rows, bool kBulk, bool kLoZero = false>
cudaError_t launch_prefill(const PrefillArgs &a, const Rows &r, cudaStream_t s) {
    switch (a.group) {
        case 1: return launch_prefill_g<1, Rows, kBulk, kLoZero>(a, r, s);
        case 2: return launch_prefill_g<2, Rows, kBulk, kLoZero>(a, r, s);
        case 4: return launch_prefill_g<4, Rows, kBulk, kLoZero>(a, r, s);
        case 8: return launch_prefill_g<8, Rows, kBulk, kLoZero>(a, r, s);
        default: return cudaErrorInvalidValue;
    }
}

// ----------------------------------------------------------- split pass ----
//
// One CTA per (row, 64-key tile, kv head): the tile's K and V rows (read once
// through the page table, widened to f32; zero past the row's keys) go to
// shared memory, then every 16-byte chunk of the four operand planes is split
// (hi = low 13 mantissa bits cleared, lo = the exact rest) and written in the
// prefill kernel's shared-memory order, chunk by chunk (coalesced).  The V
// rows are kept 129 floats apart so that reading them transposed has no bank
// conflicts.
constexpr int kSplitRawFloats = kKT * kHD + kKT * (kHD + 1);

template <class E>
__global__ void __launch_bounds__(256) split_kernel(SplitArgs p, PagedRowsP<E> rows_of) {
    // bf16 values, and fp8 values times a power of two, are exact in tf32:
    // their lo planes are zero and not written
    constexpr bool kLoZero = !std::is_same<E, float>::value;
    const float p_scale = rows_of.a.kv_scale;
    extern __shared__ __align__(16) float raw[];
    float *rk = raw;              // [64][128]
    float *rv = raw + kKT * kHD;  // [64][129]
    const int it = blockIdx.x / p.n_kv;
    const int kvh = blockIdx.x - it * p.n_kv;
    const SplitItem t = p.items[it];
    const RowDesc rd = p.rows[t.row];
    const int total_k = rd.past_len + rd.n_q;
    const int key0 = t.kt * kKT;
    // 256 threads x 8 passes = 64 keys x 32 float4 chunks; unrolled, so that
    // a thread's 16 row loads are in flight together
    static_assert(kKT * (kHD / 4) == 256 * 8, "one tile per 8 passes of 256 threads");
#pragma unroll
    for (int pass = 0; pass < 8; ++pass) {
        const int i = threadIdx.x + 256 * pass;
        const int key = i >> 5, ch = i & 31, pos = key0 + key;
        float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
        if (pos < total_k) {
            const int b = rows_of.checked(rows_of.entry(rd.slot, pos, p.err), p.err);
            if (b >= 0) {
                kx = ldg4(rows_of.k_row(b, pos, kvh) + 4 * ch);
                vx = ldg4(rows_of.v_row(b, pos, kvh) + 4 * ch);
                if constexpr (std::is_same<E, fp8>::value) {
                    const float sc = p_scale;  // power of two: exact
                    kx = make_float4(kx.x * sc, kx.y * sc, kx.z * sc, kx.w * sc);
                    vx = make_float4(vx.x * sc, vx.y * sc, vx.z * sc, vx.w * sc);
                }
            }
        }
        *reinterpret_cast<float4 *>(rk + key * kHD + 4 * ch) = kx;
        float *vd = rv + key * (kHD + 1) + 4 * ch;
        vd[0] = vx.x;
        vd[1] = vx.y;
        vd[2] = vx.z;
        vd[3] = vx.w;
    }
    __syncthreads();
    unsigned char *out = p.img + (static_cast<size_t>(t.slot) * p.n_kv + kvh) * kImageBytes;
    for (int q = threadIdx.x; q < static_cast<int>(kImagePlane / 16); q += blockDim.x) {
        float4 h, l;
        {
            // K: k-block q >> 9 (32 dims), key row (q >> 3) & 63, swizzled chunk q & 7
            const int kb = q >> 9, r = (q >> 3) & 63, lc = (q & 7) ^ (r & 7);
            split4(*reinterpret_cast<const float4 *>(rk + r * kHD + kb * 32 + lc * 4), h, l);
            *reinterpret_cast<float4 *>(out + q * 16) = h;
            if constexpr (!kLoZero) *reinterpret_cast<float4 *>(out + kImagePlane + q * 16) = l;
        }
        {
            // V^T: k-block q >> 10 (32 keys), dim row (q >> 3) & 127, swizzled chunk q & 7
            const int kb = q >> 10, d = (q >> 3) & 127, lc = (q & 7) ^ (d & 7);
            const int k0 = kb * 32 + lc * 4;
            const float4 x = make_float4(rv[k0 * (kHD + 1) + d], rv[(k0 + 1) * (kHD + 1) + d],
                                         rv[(k0 + 2) * (kHD + 1) + d], rv[(k0 + 3) * (kHD + 1) + d]);
            split4(x, h, l);
            *reinterpret_cast<float4 *>(out + 2 * kImagePlane + q * 16) = h;
            if constexpr (!kLoZero) *reinterpret_cast<float4 *>(out + 3 * kImagePlane + q * 16) = l;
        }
    }
}

template <class E>
cudaError_t launch_split(const SplitArgs &a, const PagedRowsP<E> &r, cudaStream_t s) {
    constexpr size_t smem = kSplitRawFloats * sizeof(float);
    static PerDeviceOnce configured;  // the attribute is per function and device
    const cudaError_t ce = configured.run([&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(split_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        return cudaSuccess;
    });
    if (ce != cudaSuccess) return ce;
    const long long grid = static_cast<long long>(a.n_items) * a.n_kv;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    split_kernel<E><<<static_cast<unsigned>(grid), 256, smem, s>>>(a, r);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_paged(const PrefillArgs &a, const PagedAddr &addr, cudaStream_t s) {
    // the operands come as images (whatever the pool element): one instantiation
    if (!a.img || !a.img_tile0) return cudaErrorInvalidValue;
    if (a.lo_zero) return launch_prefill<PagedRowsP<float>, true, true>(a, PagedRowsP<float>{addr}, s);
    return launch_prefill<PagedRowsP<float>, true, false>(a, PagedRowsP<float>{addr}, s);
}

cudaError_t launch_prefill_contig(const PrefillArgs &a, const ContigAddr &addr, cudaStream_t s) {
    return launch_prefill<ContigRowsP, false>(a, ContigRowsP{addr}, s);
}

cudaError_t launch_split_paged(const SplitArgs &a, const PagedAddr &addr, cudaStream_t s) {
    if (addr.fp8) return launch_split(a, PagedRowsP<fp8>{addr}, s);
    if (addr.bf16) return launch_split(a, PagedRowsP<bf16>{addr}, s);
    return launch_split(a, PagedRowsP<float>{addr}, s);
}

}  // namespace pkv
