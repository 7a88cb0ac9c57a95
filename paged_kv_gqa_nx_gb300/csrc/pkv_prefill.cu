// pkv_prefill.cu -- tensor-core attention for chunked-prefill rows (n_q > 1).
//
// For a row with many new tokens, Q.K^T over a tile of queries and keys is a
// real dense contraction, so it runs on the 5th-generation tensor cores
// (tcgen05.mma kind::f16, f32 accumulators).  To keep f32 accuracy every f32
// operand is first multiplied by a power of two (exact) that puts its largest
// magnitude in [2^14, 2^15), then split into two f16 pieces x = x0 + x1 (x0 =
// x rounded to f16, x1 = the exact rest rounded to f16: 22 significant bits),
// and every product is formed as x0*y0 + x0*y1 + x1*y0; the dropped x1*y1
// term is ~2^-22 relative.  The powers of two: one per query row, one per
// 64-key tile of K and one of V per kv head (the largest magnitude over the
// tile).  The scores are scaled back exactly before the softmax.  The
// probabilities p (at most 2^8, see the lazy rescale) of a tile whose V
// exponent is c are multiplied by 2^(C - c), where C is an exponent of the
// query tile (one per softmax chain) that only decreases and stays at most
// 7 + c for every key tile seen, so they stay at most 2^15; the accumulator
// then holds 2^C x the output's sum, is rescaled exactly when C moves, and is
// scaled back by 2^-C at the end.
//
// The K/V operands of a tile come as an image made by the split pass (below)
// from the pool's rows or from a contiguous K/V pair: the pieces already in
// the kernel's shared-memory layout, then the tile's two exponents.  Paged
// and contiguous launches read the same images of the same keys, so they
// return the same bits.
//
// One CTA = two tiles of 128 query rows of one row and one key split (two
// softmax chains that share every K/V tile); a tile is (128 / G) consecutive
// tokens x the G query heads that share kv head `kvh`.  Row m of chain c's
// tile is token m / G, head m % G, TMEM lane m and compute thread m of warps
// 4c .. 4c+3: each thread reads its row's 64 scores of a key tile, so the
// softmax needs no exchange between threads.  Warps 8 and 11 issue chain 0's
// and chain 1's QK MMAs, warp 10 the PV MMAs of both (one thread each), warp 9
// bulk-copies the images.  Key tiles are 64 positions; tile j of chain c uses
// S / P buffer j % 2 of the chain (TMEM), and K_j, V_j^T come through a ring
// of three shared-memory slots, K one tile ahead of V (K_0, K_1, V_0, K_2,
// V_1, ...):
//   QK_c(j):  S_c[128 x 64]  = Q_c.K_j^T   A = Q0_c / Q1_c (smem), B = K_j
//   PV_c(j):  D_c[128 x 128] = P_c.V_j     A = P0_c / P1_c (TMEM),  B = V_j^T
// P_c(j) is written over S_c(j) (two f16 pieces take the columns of one f32).
// QK_c(j+1) runs while the compute warps do the softmax of tile j, PV_c(j)
// after it, and the two chains' MMAs interleave on the tensor core.
// Offset-causal mask: key p visible iff p <= q_pos = total_k - n_q + i.  p is
// relative to a reference max that moves (and D is rescaled) only when a
// tile's max exceeds it by more than 2^8, which keeps every p at most 256.
// Shared memory: Q0 and Q1 of each chain (32 KiB each), three ring slots of
// 32 KiB (pieces 0, 1).  TMEM (512 columns; two f16 per column for the A
// operands): chain c's D at 128c, its S / P buffers at 256 + 128c + {0, 64}.
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
// TMEM columns: chain c's D at kColD + 128c; its S / P buffer b at
// kColSP + 128c + 64b (P piece 0 in the first 32 columns, piece 1 in the next 32)
constexpr uint32_t kColD = 0, kColSP = 256;
constexpr int kChains = 2;
constexpr int kComputeWarps = 4 * kChains;  // one thread per tile row and chain
constexpr int kWarpQK0 = 8, kWarpCopy = 9, kWarpPV = 10, kWarpQK1 = 11;
constexpr int kThreads = 32 * 12;
// registers per thread: at launch (the whole register file over the CTA),
// then the issue warpgroup (warps 8-11) after setmaxnreg.dec and the compute
// warpgroups after setmaxnreg.inc; .inc waits until the pool holds its
// registers, so the shares must add up to no more than the launch's
constexpr int kLaunchRegs = 168, kIssueRegs = 88, kComputeRegs = 208;
static_assert(kThreads * kLaunchRegs <= 65536, "launch registers exceed the register file");
static_assert(32 * kComputeWarps * kComputeRegs + 128 * kIssueRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch's registers");
constexpr float kRescale = 8.f;           // lazy-rescale threshold (base 2)
constexpr int kPExp = 7;                  // C <= kPExp + c: p * 2^(C - c) <= 2^(8 + kPExp)

// The power of two that brings a largest magnitude m into [2^14, 2^15):
// 14 - floor(log2 m), clamped to [-113, 126] (m = 0 or subnormal: 126).
__device__ __forceinline__ int f16_scale_exp(float m) {
    const int e = static_cast<int>((__float_as_uint(m) >> 23) & 255u) - 127;
    return max(-113, min(126, 14 - e));
}
// 2^n, n in [-126, 127].
__device__ __forceinline__ float pow2f(int n) { return __uint_as_float(static_cast<uint32_t>(n + 127) << 23); }
// x * 2^n, n in [-252, 254], in two exact steps (rounded only where the
// result is subnormal).
__device__ __forceinline__ float mul_pow2(float x, int n) {
    const int n1 = n / 2;
    return (x * pow2f(n1)) * pow2f(n - n1);
}
// Two f32 values (already scaled into f16's range) -> their f16 pieces, packed
// as f16 pairs (a in the low half): x0 = f16(x), x1 = f16(x - x0).
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t &p0, uint32_t &p1) {
    const __half2 h0 = __floats2half2_rn(a, b);
    const float2 f0 = __half22float2(h0);
    const __half2 h1 = __floats2half2_rn(a - f0.x, b - f0.y);
    p0 = *reinterpret_cast<const uint32_t *>(&h0);
    p1 = *reinterpret_cast<const uint32_t *>(&h1);
}
// Eight consecutive values times sc as one 16-byte chunk of each piece.
__device__ __forceinline__ void split_chunk(const float (&x)[8], float sc, uint4 &c0, uint4 &c1) {
    split_f16x2(x[0] * sc, x[1] * sc, c0.x, c1.x);
    split_f16x2(x[2] * sc, x[3] * sc, c0.y, c1.y);
    split_f16x2(x[4] * sc, x[5] * sc, c0.z, c1.z);
    split_f16x2(x[6] * sc, x[7] * sc, c0.w, c1.w);
}
__device__ __forceinline__ float absmax4(float m, const float4 &x) {
    return fmaxf(fmaxf(m, fmaxf(fabsf(x.x), fabsf(x.y))), fmaxf(fabsf(x.z), fabsf(x.w)));
}
// 2^x to about 2^-22 relative (ex2.approx; 0 for -inf and below 2^-126).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// max / sum of N values as a pairwise tree (N a power of two)
template <int N>
__device__ __forceinline__ float tree_max(const float (&v)[N]) {
    float t[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) t[i] = fmaxf(v[2 * i], v[2 * i + 1]);
#pragma unroll
    for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = fmaxf(t[2 * i], t[2 * i + 1]);
    return t[0];
}
template <int N>
__device__ __forceinline__ float tree_sum(const float (&v)[N]) {
    float t[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) t[i] = v[2 * i] + v[2 * i + 1];
#pragma unroll
    for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = t[2 * i] + t[2 * i + 1];
    return t[0];
}

// Rows of the split pass: through the page table, or a contiguous K/V pair.
template <class E>
struct PagedRowsP {
    using Elem = E;
    PagedAddr a;
    // The page-table entry of (slot, pos): -1 when the page index is out of
    // range (error flag set), else the raw entry, which checked() validates.
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
    __device__ __forceinline__ float scale() const { return a.kv_scale; }
};

struct ContigRowsP {
    using Elem = float;
    ContigAddr a;
    __device__ __forceinline__ int entry(int, int, int32_t *) const { return 0; }
    __device__ __forceinline__ int checked(int blk, int32_t *) const { return blk; }
    __device__ __forceinline__ const float *k_row(int, int pos, int kvh) const {
        return a.k + static_cast<size_t>(pos) * a.kv_dim + static_cast<size_t>(kvh) * kHD;
    }
    __device__ __forceinline__ const float *v_row(int, int pos, int kvh) const {
        return a.v + static_cast<size_t>(pos) * a.kv_dim + static_cast<size_t>(kvh) * kHD;
    }
    __device__ __forceinline__ float scale() const { return 1.f; }
};

constexpr uint32_t kSmemQ = 64 * 1024;  // one chain's Q0, Q1: each 2 k-blocks of 128 rows x 64 f16
// one ring slot: pieces 0, 1 of K_j (each 2 k-blocks of 64 rows x 64 f16) or
// of V_j^T (each 1 k-block of 128 rows x 64 f16)
constexpr uint32_t kSmemKV = 2 * kImagePlane;
static_assert(kImagePlane == 16 * 1024, "a piece of a tile is 16 KiB");
constexpr int kSlots = 3;
constexpr size_t kSmemBytes = kChains * kSmemQ + kSlots * kSmemKV + 1024;  // + alignment slack

// kLoZero (images of a bf16 or fp8 pool): the K / V piece-1 planes are left
// out -- a pool value times the tile's power of two is exact in f16 unless it
// lies more than 2^28 below the tile's largest magnitude, where it is rounded
// to an f16 subnormal (an error below 2^-38 of that magnitude) -- so they are
// neither copied nor used.
//
// mbarriers.  Ring item i sits in slot i % 3, phase (i / 3) % 2:
//   full[s]    the item's bytes landed (the copy warp's expect-tx arrival)
//   free[s]    every MMA that reads the item complete: two commits, one per
//              QK warp for a K item, both from the PV warp for a V item
// Per chain c and S / P buffer b, phase (j / 2) % 2 for tile j (qready: once):
//   qready[c]     Q_c written (compute warps of chain c)
//   sdone[c][b]   QK_c(j) complete (commit): S_c(j) readable
//   pready[c][b]  P_c(j) written over S_c(j) (compute warps)
//   pvdone[c][b]  PV_c(j) complete (commit): the buffer free for QK_c(j+2)
// The MMAs are issued by three warps, and a QK warp takes every wait of a
// tile before its first MMA: a thread's mbarrier test after its own MMAs
// waits for them to reach the tensor core, so a wait between MMAs drains the
// tensor pipe unless another warp's MMAs are queued.  No waiter is ever two phases behind: each next phase needs an
// arrival that follows the wait.
template <int G, bool kLoZero>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(PrefillArgs a) {
    constexpr int TQ = 128 / G;  // tokens per tile
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *Qs = sm;                       // chain c: Q0 at c * kSmemQ, Q1 32 KiB on
    unsigned char *ring = Qs + kChains * kSmemQ;  // slot s at s * kSmemKV: pieces 0, 1 (+ kImagePlane)
    __shared__ uint64_t bar_full[kSlots], bar_free[kSlots];
    __shared__ uint64_t bar_qready[kChains], bar_sdone[kChains][2], bar_pready[kChains][2], bar_pvdone[kChains][2];
    __shared__ uint32_t tslot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pi = blockIdx.x / a.n_kv;
    const int kvh = blockIdx.x - pi * a.n_kv;
    // the pair's tiles: one row and one split; the second may be absent
    const PrefillTile t0 = a.tiles[2 * pi], t1 = a.tiles[2 * pi + 1];
    const RowDesc rd = a.rows[t0.row];
    const int total_k = rd.past_len + rd.n_q;
    const int kbeg = t0.split * a.split_keys;
    const int kt0 = kbeg / kKT;
    // a tile's end within the split (kend: its last visible key + 1, at
    // most the split's end) and its key tiles
    auto tile_keys = [&](const PrefillTile &t, int &kend) {
        const int n_valid_q = min(TQ, rd.n_q - t.q0);
        const int kend_tile = a.causal ? min(total_k, total_k - rd.n_q + t.q0 + n_valid_q) : total_k;
        kend = min(kbeg + a.split_keys, kend_tile);
        return max(0, (kend + kKT - 1) / kKT - kt0);
    };
    int kend0, kend1 = 0;
    const int n0 = tile_keys(t0, kend0);
    int n1 = 0;
    if (t1.row >= 0) {
        if (t1.row == t0.row && t1.split == t0.split) {
            n1 = tile_keys(t1, kend1);
        } else if (tid == 0 && a.err) {
            atomicOr(a.err, 1);  // not a pair: the second tile is dropped
        }
    }
    const int n_max = max(n0, n1);  // key tiles loaded
    auto ph = [](int j) { return static_cast<uint32_t>(j >> 1) & 1u; };        // buffer j % 2
    auto rph = [](int i) { return static_cast<uint32_t>(i / kSlots) & 1u; };  // ring item i
    // ring items: K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}
    auto k_item = [](int j) { return j == 0 ? 0 : 2 * j - 1; };
    auto v_item = [&](int j) { return j + 1 < n_max ? 2 * j + 2 : 2 * j + 1; };
    // lane 0 waits (bounded), the warp learns the outcome
    auto wait_w = [&](uint64_t *bar, uint32_t parity) {
        return __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(smem_u32(bar), parity) : true, 0) != 0;
    };

    if (warp == 0) {
        tmem_alloc(smem_u32(&tslot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int sl = 0; sl < kSlots; ++sl) {
            mbar_init(smem_u32(&bar_full[sl]), 1);  // the copy warp's expect-tx arrival
            mbar_init(smem_u32(&bar_free[sl]), 2);
        }
        for (int c = 0; c < kChains; ++c) {
            mbar_init(smem_u32(&bar_qready[c]), 4);  // the chain's four compute warps
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&bar_sdone[c][b]), 1);
                mbar_init(smem_u32(&bar_pready[c][b]), 4);
                mbar_init(smem_u32(&bar_pvdone[c][b]), 1);
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;
    bool ok = true;
    const int32_t *slots = a.img_slot + a.img_tile0[t0.row];  // images of the row's key tiles
    auto image = [&](int32_t slot) {
        return a.img + (static_cast<size_t>(slot) * a.n_kv + kvh) * kImageBytes;
    };

    if (warp >= kComputeWarps) {
        setmaxnreg_dec<kIssueRegs>();
        if (warp == kWarpCopy) {
            // ---------------- copy warp (lane 0 copies) ----------------
            // Ring item i is copied as soon as the MMAs that read item i - 3
            // (the slot's previous item) are done; each copy arrives with its
            // byte count on the slot's full barrier.  Item i: K_0 (i = 0),
            // V_{n-1} (the last), else K_{(i+1)/2} (odd i) or V_{(i-2)/2}.
            constexpr uint32_t planes = kLoZero ? 1u : 2u;  // pieces 0 (and 1) of K / V
            int issued = 0;
            for (int i = 0; i < 2 * n_max; ++i) {
                const int sl = i % kSlots;
                if (i >= kSlots && !wait_w(&bar_free[sl], rph(i - kSlots))) break;
                const bool is_v = i > 0 && ((i & 1) == 0 || i == 2 * n_max - 1);
                const int jt = i == 0 ? 0 : (i == 2 * n_max - 1 ? n_max - 1 : ((i & 1) ? (i + 1) >> 1 : (i - 2) >> 1));
                if (lane == 0) {
                    // K_j: planes 0, 1 of the image; V_j^T: planes 2, 3
                    const unsigned char *src = image(__ldg(slots + kt0 + jt)) + (is_v ? 2 : 0) * kImagePlane;
                    unsigned char *dst = ring + sl * kSmemKV;
                    mbar_expect_tx(smem_u32(&bar_full[sl]), planes * kImagePlane);
                    bulk_g2s(smem_u32(dst), src, kImagePlane, smem_u32(&bar_full[sl]));
                    if constexpr (planes == 2)
                        bulk_g2s(smem_u32(dst + kImagePlane), src + kImagePlane, kImagePlane,
                                 smem_u32(&bar_full[sl]));
                }
                issued = i + 1;
            }
            // let the last copies land before the CTA's shared memory is given
            // up (every earlier one was waited for before its slot was
            // refilled; bounded if the other warps gave up)
            for (int i = max(0, issued - kSlots); i < issued; ++i) wait_w(&bar_full[i % kSlots], rph(i));
        } else if (warp == kWarpQK0 || warp == kWarpQK1) {
            // ---------- QK issue warps (lane 0 issues): QK_c(j) ----------
            // one k-step (16 dims): three products of the pieces (the one with
            // the K piece-1 plane is left out when that plane is zero).  Every
            // K item gets one commit from each QK warp, also past the chain's
            // last tile (after the item landed, so that it counts for its
            // own phase).
            constexpr bool lo = !kLoZero;
            const int c = warp == kWarpQK1 ? 1 : 0;
            const int n = c ? n1 : n0;
            const uint32_t idesc_s = idesc_f16(128, kKT);
            const uint64_t dQ0 = desc_sw128(smem_u32(Qs + c * kSmemQ));
            const uint64_t dQ1 = desc_sw128(smem_u32(Qs + c * kSmemQ + kSmemQ / 2));
            for (int j = 0; j < n_max && ok; ++j) {
                const int b = j & 1, i = k_item(j), sl = i % kSlots;
                // every wait of the tile first: K_j landed, the chain's S / P
                // buffer free (PV_c(j-2) done) and, for tile 0, its Q written
                ok = wait_w(&bar_full[sl], rph(i));
                if (ok && j < n) {
                    if (j == 0) ok = wait_w(&bar_qready[c], 0);
                    else if (j >= 2) ok = wait_w(&bar_pvdone[c][b], ph(j - 2));
                }
                if (!ok) break;
                fence_after_sync();
                if (lane == 0) {
                    if (j < n) {
                        const uint64_t dK0 = desc_sw128(smem_u32(ring + sl * kSmemKV));
                        const uint64_t dK1 = desc_sw128(smem_u32(ring + sl * kSmemKV + kImagePlane));
                        const uint32_t tS = tbase + kColSP + 128u * c + 64u * b;
#pragma unroll
                        for (int s = 0; s < kHD / 16; ++s) {
                            const uint64_t ko = ((s >> 2) * 8192u + (s & 3) * 32u) >> 4;
                            const uint64_t qo = ((s >> 2) * 16384u + (s & 3) * 32u) >> 4;
                            mma_f16(tS, dQ0 + qo, dK0 + ko, idesc_s, s > 0);
                            if constexpr (lo) mma_f16(tS, dQ0 + qo, dK1 + ko, idesc_s, 1);
                            mma_f16(tS, dQ1 + qo, dK0 + ko, idesc_s, 1);
                        }
                        mma_commit(smem_u32(&bar_sdone[c][b]));
                    }
                    mma_commit(smem_u32(&bar_free[sl]));
                }
                __syncwarp();
            }
            if (!ok && lane == 0 && a.err) atomicOr(a.err, 2);
        } else if (warp == kWarpPV) {
            // ---------- PV issue warp (lane 0 issues): PV_0(j), PV_1(j) ----------
            constexpr bool lo = !kLoZero;
            const uint32_t idesc_o = idesc_f16(128, kHD);
            for (int j = 0; j < n_max && ok; ++j) {
                const int b = j & 1, i = v_item(j), sl = i % kSlots;
                ok = wait_w(&bar_full[sl], rph(i));
                if (!ok) break;
                const uint64_t dV0 = desc_sw128(smem_u32(ring + sl * kSmemKV));
                const uint64_t dV1 = desc_sw128(smem_u32(ring + sl * kSmemKV + kImagePlane));
#pragma unroll 1
                for (int c = 0; c < kChains; ++c) {
                    if (j >= (c ? n1 : n0)) continue;
                    ok = wait_w(&bar_pready[c][b], ph(j));
                    if (!ok) break;
                    fence_after_sync();
                    if (lane == 0) {
                        const uint32_t tP = tbase + kColSP + 128u * c + 64u * b, tD = tbase + kColD + 128u * c;
#pragma unroll
                        for (int s = 0; s < kKT / 16; ++s) {
                            const uint64_t vo = (s * 32u) >> 4;
                            mma_f16_ts(tD, tP + 8 * s, dV0 + vo, idesc_o, j > 0 || s > 0);
                            if constexpr (lo) mma_f16_ts(tD, tP + 8 * s, dV1 + vo, idesc_o, 1);
                            mma_f16_ts(tD, tP + 32 + 8 * s, dV0 + vo, idesc_o, 1);
                        }
                        mma_commit(smem_u32(&bar_pvdone[c][b]));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) {  // the V item's two arrivals
                    mma_commit(smem_u32(&bar_free[sl]));
                    mma_commit(smem_u32(&bar_free[sl]));
                }
                __syncwarp();
            }
            if (!ok && lane == 0 && a.err) atomicOr(a.err, 2);
        }
    } else {
        // -------------- compute warps: one thread per tile row and chain --------------
        setmaxnreg_inc<kComputeRegs>();
        const int c = warp >> 2;  // chain
        const int n = c ? n1 : n0;
        const int q0 = c ? t1.q0 : t0.q0, kend = c ? kend1 : kend0;
        const uint32_t cD = kColD + 128u * c, cSP = kColSP + 128u * c;
        unsigned char *Q0 = Qs + c * kSmemQ, *Q1 = Q0 + kSmemQ / 2;
        const int m = tid & 127;  // this thread's row of the tile (TMEM lane)
        const int tq = m / G, g = m - (m / G) * G;
        const int qi = q0 + tq;
        const bool valid = qi < rd.n_q;
        const int q_pos = total_k - rd.n_q + qi;
        const int kend_row = valid ? (a.causal ? min(q_pos + 1, total_k) : total_k) : 1;
        const int klim = min(kend_row, kend);  // keys below klim are visible to this row
        const uint32_t tlane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        // this warp's arrival on a barrier, after its TMEM stores
        auto arrive = [&](uint64_t *bar) {
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(bar));
        };

        if (n > 0) {
            // Q row (pre-scaled to base-2 units, then by the row's power of
            // two) -> its two pieces in shared memory.  All 32 loads of the row
            // are issued together (one memory latency), then its largest
            // magnitude, then the pieces.
            int qexp;
            {
                const float4 *qrow = reinterpret_cast<const float4 *>(
                    a.Q + static_cast<size_t>(rd.q_row0 + (valid ? qi : 0)) * (a.n_heads * kHD) +
                    static_cast<size_t>(kvh * G + g) * kHD);
                float4 q[kHD / 4];
#pragma unroll
                for (int j4 = 0; j4 < kHD / 4; ++j4)
                    q[j4] = valid ? __ldg(qrow + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
                float mx = 0.f;
#pragma unroll
                for (int j4 = 0; j4 < kHD / 4; ++j4) {
                    q[j4].x *= a.scale_log2;
                    q[j4].y *= a.scale_log2;
                    q[j4].z *= a.scale_log2;
                    q[j4].w *= a.scale_log2;
                    mx = absmax4(mx, q[j4]);
                }
                qexp = f16_scale_exp(mx);
                const float qs = pow2f(qexp);
#pragma unroll
                for (int cc = 0; cc < kHD / 8; ++cc) {  // dims 8cc .. 8cc + 7: k-block cc / 8, chunk cc % 8
                    const float x[8] = {q[2 * cc].x,     q[2 * cc].y,     q[2 * cc].z,     q[2 * cc].w,
                                        q[2 * cc + 1].x, q[2 * cc + 1].y, q[2 * cc + 1].z, q[2 * cc + 1].w};
                    uint4 c0, c1;
                    split_chunk(x, qs, c0, c1);
                    const uint32_t off = (cc >> 3) * 16384u + sw128_chunk(m, cc & 7);
                    *reinterpret_cast<uint4 *>(Q0 + off) = c0;
                    *reinterpret_cast<uint4 *>(Q1 + off) = c1;
                }
            }
            fence_proxy_async();  // generic-proxy writes, before the MMAs read them
            arrive(&bar_qready[c]);

            // The output accumulator lives in TMEM (D) and the P.V MMAs add into
            // it.  p is taken relative to a reference max m_ref that moves only
            // when a tile's max exceeds it by more than kRescale (base-2 units);
            // then D and l are rescaled once.
            float m_ref = -INFINITY, l_run = 0.f;
            int cexp = 0;  // C: D holds 2^C x the output's sum
            // the tile exponents (K, V), read from the images a tile ahead
            int2 ex_cur = __ldg(reinterpret_cast<const int2 *>(image(__ldg(slots + kt0)) + kImageExpOff));
            int32_t slot_next = n > 1 ? __ldg(slots + kt0 + 1) : 0;

            for (int j = 0; j < n; ++j) {
                const int kt = kt0 + j, b = j & 1;
                const uint32_t tSP = tbase + tlane + cSP + 64u * b;
                // S_c(j) ready (QK_c(j) done)
                ok = wait_w(&bar_sdone[c][b], ph(j));
                if (!ok) break;
                fence_after_sync();
                float s[kKT];
                {
                    float h[32];
                    tmem_ld32(tSP, h);
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[i] = h[i];
                    tmem_ld32(tSP + 32, h);
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[32 + i] = h[i];
                }
                const int kexp = ex_cur.x, vexp = ex_cur.y;

                // scores to base-2 units: one exact factor 2^sn (two steps when
                // 2^sn is not a normal f32); mask the keys this row does not see
                const int sn = -(qexp + kexp);
                const bool one = sn >= -126 && sn <= 127;
                const float fsc = one ? pow2f(sn) : 1.f;
                if (!one) {
                    const float sa = pow2f(sn / 2), sb = pow2f(sn - sn / 2);
#pragma unroll
                    for (int i = 0; i < kKT; ++i) s[i] = (s[i] * sa) * sb;
                }
                const int base = kt * kKT;
                if (base + kKT > klim) {
#pragma unroll
                    for (int i = 0; i < kKT; ++i) s[i] = base + i < klim ? s[i] : -INFINITY;
                }
                const float row_max = tree_max(s) * fsc;
                const bool rescale = m_ref != -INFINITY && row_max > m_ref + kRescale;
                const float m_use = (m_ref == -INFINITY || rescale) ? row_max : m_ref;
                // p = 2^(s - m_use): one FFMA (exact scaling, one rounding) and ex2
                const float nm = m_use == -INFINITY ? 0.f : -m_use;
#pragma unroll
                for (int i = 0; i < kKT; ++i) s[i] = ex2_approx(fmaf(s[i], fsc, nm));
                const float rowsum = tree_sum(s);
                // C for this tile (the same in every thread of the chain)
                const int c_new = j == 0 ? kPExp + vexp : min(cexp, kPExp + vexp);

                // D moves (a row's reference max, or C): PV_c(j-1) done first;
                // tcgen05.ld / st are warp-collective, so the whole warp takes
                // the branch (rows that do not rescale multiply by 2^(C'-C))
                const bool cmove = j > 0 && c_new != cexp;
                const float f = rescale ? exp2f(m_ref - m_use) : 1.f;
                if (cmove || __any_sync(0xffffffffu, rescale)) {
                    ok = wait_w(&bar_pvdone[c][b ^ 1], ph(j - 1));
                    if (!ok) break;
                    fence_after_sync();
                    const float fd = mul_pow2(f, c_new - cexp);
#pragma unroll
                    for (int cc = 0; cc < kHD / 16; ++cc) {  // 16 columns at a time: the scores are live
                        float dv[16];
                        tmem_ld16(tbase + tlane + cD + 16 * cc, dv);
#pragma unroll
                        for (int i = 0; i < 16; ++i) dv[i] *= fd;
                        tmem_st16(tbase + tlane + cD + 16 * cc, dv);
                    }
                }
                l_run = l_run * f + rowsum;
                m_ref = m_use;
                cexp = c_new;

                // P_j * 2^(C - c) over S as two f16 pieces; the PV warp starts PV_c(j)
                {
                    const int pe = cexp - vexp;  // <= kPExp
                    const float pf = pe >= -126 ? pow2f(pe) : 0.f;
                    uint32_t p0[32], p1[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) split_f16x2(s[2 * i] * pf, s[2 * i + 1] * pf, p0[i], p1[i]);
                    tmem_st32u(tSP, p0);
                    tmem_st32u(tSP + 32, p1);
                }
                arrive(&bar_pready[c][b]);

                // the next tile's exponents
                if (j + 1 < n) {
                    ex_cur = __ldg(reinterpret_cast<const int2 *>(image(slot_next) + kImageExpOff));
                    if (j + 2 < n) slot_next = __ldg(slots + kt + 2);
                }
            }
            // the last PV, then the result: D / l, then * 2^-C (exact); in that
            // order the output does not overflow where D * 2^-C (up to l times
            // it) would
            if (ok) ok = wait_w(&bar_pvdone[c][(n - 1) & 1], ph(n - 1));
            if (!ok) {
                if (lane == 0 && a.err) atomicOr(a.err, 2);
            } else {
                fence_after_sync();
                // the tile's output placement, read again here rather than
                // held through the loop
                const PrefillTile tile = a.tiles[2 * pi + c];
                const int h = kvh * G + g;
                const bool direct = tile.part0 < 0;
                float *dst = nullptr;
                size_t pidx = 0;
                if (direct) {
                    dst = a.out + static_cast<size_t>(rd.q_row0 + (valid ? qi : 0)) * (a.n_heads * kHD) +
                          static_cast<size_t>(h) * kHD;
                } else {
                    const int n_valid_q = min(TQ, rd.n_q - tile.q0);
                    const int kend_tile =
                        a.causal ? min(total_k, total_k - rd.n_q + tile.q0 + n_valid_q) : total_k;
                    const int n_split = (kend_tile + a.split_keys - 1) / a.split_keys;
                    const int stride = tile.stride > 0 ? tile.stride : n_split;
                    pidx = static_cast<size_t>(tile.part0 + (valid ? tq : 0) * stride + tile.split) * a.n_heads + h;
                    dst = a.pacc + pidx * kHD;
                }
                const float scl = direct ? 1.f / l_run : 1.f;
#pragma unroll
                for (int cc = 0; cc < kHD / 32; ++cc) {
                    float dv[32];
                    tmem_ld32(tbase + tlane + cD + 32 * cc, dv);
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(dst + 32 * cc + i) =
                                make_float4(mul_pow2(dv[i] * scl, -cexp), mul_pow2(dv[i + 1] * scl, -cexp),
                                            mul_pow2(dv[i + 2] * scl, -cexp), mul_pow2(dv[i + 3] * scl, -cexp));
                    }
                }
                if (valid && !direct) {
                    a.pm[pidx] = m_ref;
                    a.pl[pidx] = l_run;
                }
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

template <int G, bool kLoZero>
cudaError_t launch_prefill_g(const PrefillArgs &a, cudaStream_t s) {
    static PerDeviceOnce configured;  // the attributes are per function and device
    const cudaError_t ce = configured.run([&]() -> cudaError_t {
        // setmaxnreg.inc waits until the CTA's pool holds the registers asked
        // for, so launch only if the compiled kernel starts with the registers
        // the split was sized for
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<G, kLoZero>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < kLaunchRegs || fa.maxThreadsPerBlock < kThreads) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(prefill_tc_kernel<G, kLoZero>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemBytes));
    });
    if (ce != cudaSuccess) return ce;
    // two tiles per CTA
    if (a.n_tiles <= 0 || (a.n_tiles & 1)) return cudaErrorInvalidValue;
    const long long grid = static_cast<long long>(a.n_tiles / 2) * a.n_kv;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prefill_tc_kernel<G, kLoZero><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, s>>>(a);
    return cudaGetLastError();
}

template <bool kLoZero>
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t s) {
    if (!a.img || !a.img_tile0 || !a.img_slot) return cudaErrorInvalidValue;
    switch (a.group) {
        case 1: return launch_prefill_g<1, kLoZero>(a, s);
        case 2: return launch_prefill_g<2, kLoZero>(a, s);
        case 4: return launch_prefill_g<4, kLoZero>(a, s);
        case 8: return launch_prefill_g<8, kLoZero>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

// ----------------------------------------------------------- split pass ----
//
// Two CTAs per (row, 64-key tile, kv head), one for K and one for V: the
// tile's rows of that operand (read once, through the page table or from a
// contiguous pair, widened to f32, an fp8 pool's scale applied; zero past the
// row's keys) go to shared memory, and the block finds their largest
// magnitude; then every 16-byte chunk of the operand's two planes is written
// in the prefill kernel's shared-memory order, chunk by chunk (coalesced):
// eight values times the tile's power of two, split into their two f16
// pieces, and the operand's exponent after the planes.  V rows are kept 129
// floats apart so that reading them transposed has no bank conflicts.  One
// operand per CTA halves the staging, so twice as many CTAs share an SM.
constexpr int kSplitRawFloats = kKT * (kHD + 1);

template <class Rows>
__global__ void __launch_bounds__(256) split_kernel(SplitArgs p, Rows rows_of) {
    using E = typename Rows::Elem;
    // a bf16 / fp8 value times a power of two is exact in f16 (but for
    // values more than 2^28 below the tile's largest): the piece-1 planes are
    // not written
    constexpr bool kLoZero = !std::is_same<E, float>::value;
    extern __shared__ __align__(16) float raw[];
    __shared__ float wmax[8];
    const int part = blockIdx.x & 1;  // 0: K, 1: V
    const int ik = blockIdx.x >> 1;
    const int it = ik / p.n_kv;
    const int kvh = ik - it * p.n_kv;
    const SplitItem t = p.items[it];
    const RowDesc rd = p.rows[t.row];
    const int total_k = rd.past_len + rd.n_q;
    const int key0 = t.kt * kKT;
    const int ld = part ? kHD + 1 : kHD;  // row pitch in shared memory
    float mx = 0.f;
    // 256 threads x 8 passes = 64 keys x 32 float4 chunks; unrolled, so that
    // a thread's 8 row loads are in flight together
    static_assert(kKT * (kHD / 4) == 256 * 8, "one tile per 8 passes of 256 threads");
#pragma unroll
    for (int pass = 0; pass < 8; ++pass) {
        const int i = threadIdx.x + 256 * pass;
        const int key = i >> 5, ch = i & 31, pos = key0 + key;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (pos < total_k) {
            const int b = rows_of.checked(rows_of.entry(rd.slot, pos, p.err), p.err);
            if (b >= 0) {
                x = ldg4((part ? rows_of.v_row(b, pos, kvh) : rows_of.k_row(b, pos, kvh)) + 4 * ch);
                if constexpr (std::is_same<E, fp8>::value) {
                    const float sc = rows_of.scale();  // power of two: exact
                    x = make_float4(x.x * sc, x.y * sc, x.z * sc, x.w * sc);
                }
            }
        }
        mx = absmax4(mx, x);
        float *d = raw + key * ld + 4 * ch;
        if (part) {
            d[0] = x.x;
            d[1] = x.y;
            d[2] = x.z;
            d[3] = x.w;
        } else {
            *reinterpret_cast<float4 *>(d) = x;
        }
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = wmax[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, wmax[w]);
    const int ex = f16_scale_exp(mx);
    const float sc = pow2f(ex);
    unsigned char *out = p.img + (static_cast<size_t>(t.slot) * p.n_kv + kvh) * kImageBytes +
                         static_cast<size_t>(part) * 2 * kImagePlane;
    for (int q = threadIdx.x; q < static_cast<int>(kImagePlane / 16); q += blockDim.x) {
        uint4 c0, c1;
        float x[8];
        if (part == 0) {
            // K: k-block q >> 9 (64 dims), key row (q >> 3) & 63, swizzled chunk q & 7
            const int kb = q >> 9, r = (q >> 3) & 63, lc = (q & 7) ^ (r & 7);
            const float *src = raw + r * kHD + kb * 64 + lc * 8;
            const float4 a0 = *reinterpret_cast<const float4 *>(src);
            const float4 a1 = *reinterpret_cast<const float4 *>(src + 4);
            x[0] = a0.x;
            x[1] = a0.y;
            x[2] = a0.z;
            x[3] = a0.w;
            x[4] = a1.x;
            x[5] = a1.y;
            x[6] = a1.z;
            x[7] = a1.w;
        } else {
            // V^T: dim row q >> 3, swizzled chunk q & 7 (8 keys)
            const int d = q >> 3, k0 = ((q & 7) ^ (d & 7)) * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = raw[(k0 + j) * (kHD + 1) + d];
        }
        split_chunk(x, sc, c0, c1);
        *reinterpret_cast<uint4 *>(out + q * 16) = c0;
        if constexpr (!kLoZero) *reinterpret_cast<uint4 *>(out + kImagePlane + q * 16) = c1;
    }
    if (threadIdx.x == 0) {
        int32_t *e = reinterpret_cast<int32_t *>(p.img + (static_cast<size_t>(t.slot) * p.n_kv + kvh) * kImageBytes +
                                                 kImageExpOff);
        e[part] = ex;
    }
}

template <class Rows>
cudaError_t launch_split(const SplitArgs &a, const Rows &r, cudaStream_t s) {
    constexpr size_t smem = kSplitRawFloats * sizeof(float);
    static PerDeviceOnce configured;  // the attribute is per function and device
    const cudaError_t ce = configured.run([&]() -> cudaError_t {
        return cudaFuncSetAttribute(split_kernel<Rows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    if (ce != cudaSuccess) return ce;
    const long long grid = static_cast<long long>(a.n_items) * a.n_kv * 2;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    split_kernel<Rows><<<static_cast<unsigned>(grid), 256, smem, s>>>(a, r);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_paged(const PrefillArgs &a, const PagedAddr &, cudaStream_t s) {
    return a.lo_zero ? launch_prefill<true>(a, s) : launch_prefill<false>(a, s);
}

cudaError_t launch_prefill_contig(const PrefillArgs &a, const ContigAddr &, cudaStream_t s) {
    return launch_prefill<false>(a, s);
}

cudaError_t launch_split_paged(const SplitArgs &a, const PagedAddr &addr, cudaStream_t s) {
    if (addr.fp8) return launch_split(a, PagedRowsP<fp8>{addr}, s);
    if (addr.bf16) return launch_split(a, PagedRowsP<bf16>{addr}, s);
    return launch_split(a, PagedRowsP<float>{addr}, s);
}

cudaError_t launch_split_contig(const SplitArgs &a, const ContigAddr &addr, cudaStream_t s) {
    return launch_split(a, ContigRowsP{addr}, s);
}

}  // namespace pkv
