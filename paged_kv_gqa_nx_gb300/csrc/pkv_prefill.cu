// pkv_prefill.cu -- tensor-core attention for chunked-prefill rows (n_q > 1).
//
// For a row with many new tokens, Q.K^T over a tile of queries and keys is a
// real dense contraction, so it runs on the 5th-generation tensor cores
// (tcgen05.mma kind::tf32).  To keep f32 accuracy each f32 operand x is split
// into a tf32 part and its exact f32 rest (x = hi + lo) and every product is
// formed as hi*hi + hi*lo + lo*hi; the dropped lo*lo term is ~2^-20 relative.
//
// One CTA = one tile of 128 query rows -- (128 / G) consecutive tokens x the G
// query heads that share kv head `kvh` -- and one key split; 256 threads.
// Row m of the tile is token m / G, head m % G and TMEM lane m; the two
// threads that share TMEM lane m (warps w and w + 4) each own 32 of a key
// tile's scores and half of the row's output columns, and exchange the row
// max and sum through shared memory.  Two threads issue the MMAs (QK and PV
// concurrently, each committing to its own mbarrier).  Key tiles are 64
// positions:
//   QK(j):  S[128 x 64]  = Q.K_j^T     A = Q hi (TMEM) / Q lo (smem), B = K_j (smem)
//   PV(j):  D[128 x 128] = P_j.V_j     A = P hi/lo (TMEM),            B = V_j^T (smem)
// Loop j: wait S_j -> online softmax (offset-causal mask: key p visible iff
// p <= q_pos = total_k - n_q + i) -> wait PV(j-1) -> write P_j, V_j, K_{j+1}
// -> QK(j+1) and PV(j) are issued, PV adding into the TMEM
// accumulator D; the softmax of tile j+1 runs while PV(j) executes.  p is
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
#include "pkv_internal.h"
#include "pkv_tcgen05.h"

namespace pkv {
namespace {

using namespace tc;

constexpr int kHD = 128;
constexpr int kKT = 64;  // keys per tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQhi = 0, kColS = 128, kColPhi = 256, kColPlo = 320, kColD = 384;
constexpr int kThreads = 256;                 // two threads per tile row
constexpr float kRescale = 8.f;               // lazy-rescale threshold (base 2)

struct PagedRowsP {
    PagedAddr a;
    __device__ __forceinline__ bool row(int slot, int pos, int kvh, const float *&kr,
                                        const float *&vr, int32_t *err) const {
        const int bi = a.bs_shift >= 0 ? (pos >> a.bs_shift) : (pos / a.bs);
        const int off = pos - bi * a.bs;
        if (bi >= a.max_blocks) {
            if (err) atomicOr(err, 1);
            return false;
        }
        const int blk = __ldg(a.pt + static_cast<size_t>(slot) * a.max_blocks + bi);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.n_blocks)) {
            if (err) atomicOr(err, 1);
            return false;
        }
        const size_t o = static_cast<size_t>(blk) * a.block_stride + a.layer_off +
                         static_cast<size_t>(off) * a.kv_dim + static_cast<size_t>(kvh) * kHD;
        kr = a.k + o;
        vr = a.v + o;
        return true;
    }
    // groups of 8 positions starting at a multiple of 8 lie in one block
    __device__ __forceinline__ bool whole8() const { return (a.bs & 7) == 0; }
    __device__ __forceinline__ size_t row_stride() const { return static_cast<size_t>(a.kv_dim); }
};

struct ContigRowsP {
    ContigAddr a;
    __device__ __forceinline__ bool row(int, int pos, int kvh, const float *&kr, const float *&vr,
                                        int32_t *) const {
        const size_t o = static_cast<size_t>(pos) * a.kv_dim + static_cast<size_t>(kvh) * kHD;
        kr = a.k + o;
        vr = a.v + o;
        return true;
    }
    __device__ __forceinline__ bool whole8() const { return true; }
    __device__ __forceinline__ size_t row_stride() const { return static_cast<size_t>(a.kv_dim); }
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

template <int G, class Rows>
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
    __shared__ uint64_t bar_qk, bar_pv;
    __shared__ uint32_t tslot;
    __shared__ float red[2][kThreads];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, half = (warp >> 2) & 1;  // TMEM lane quadrant, key / column half
    const int m = 32 * wq + lane;                      // this thread's row of the tile
    const int ti = blockIdx.x / a.n_kv;
    const int kvh = blockIdx.x - ti * a.n_kv;
    const PrefillTile tile = a.tiles[ti];
    const RowDesc rd = a.rows[tile.row];
    const int total_k = rd.past_len + rd.n_q;

    const int tq = m / G, g = m - (m / G) * G;
    const int qi = tile.q0 + tq;
    const bool valid = qi < rd.n_q;
    const int q_pos = total_k - rd.n_q + qi;
    const int kend_row = valid ? (a.causal ? min(q_pos + 1, total_k) : total_k) : 1;

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
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;
    bool ok = true;

    {
        // ---- compute warps ----
        const uint32_t tlane = static_cast<uint32_t>(32 * wq) << 16;
        // Q row (pre-scaled to base-2 units): hi -> TMEM, lo -> smem (A operands)
        {
            const float *qrow = a.Q + static_cast<size_t>(rd.q_row0 + (valid ? qi : 0)) * (a.n_heads * kHD) +
                                static_cast<size_t>(kvh * G + g) * kHD + 64 * half;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float hv[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    float4 x = valid ? __ldg(reinterpret_cast<const float4 *>(qrow + 32 * c) + j4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
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
                    const uint32_t off = (2 * half + c) * 16384u + sw128_chunk(m, j4);
                    *reinterpret_cast<float4 *>(Qlo + off) = l;
                }
                tmem_st32(tbase + tlane + kColQhi + 64 * half + 32 * c, hv);
            }
        }

        // K rows key-major (8 keys per warp, one 512-byte row per instruction;
        // one page-table lookup per warp when a block holds whole 8-key groups),
        // V rows key-per-lane for the transposed store
        float4 kreg[8], vreg[8];
        const bool k_whole = rows_of.whole8();
        const size_t rstride = rows_of.row_stride();
        auto prefetch_k = [&](int kt) {
            const int pos0 = kt * kKT + warp * 8;
            if (k_whole) {
                const float *kr, *vr;
                const bool have = pos0 < kend && rows_of.row(rd.slot, pos0, kvh, kr, vr, a.err);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    kreg[i] = (have && pos0 + i < kend)
                                  ? __ldg(reinterpret_cast<const float4 *>(kr + i * rstride) + lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float *kr, *vr;
                    const bool have = pos0 + i < kend && rows_of.row(rd.slot, pos0 + i, kvh, kr, vr, a.err);
                    kreg[i] = have ? __ldg(reinterpret_cast<const float4 *>(kr) + lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        };
        auto prefetch_v = [&](int kt) {
            const int pos = kt * kKT + 32 * half + lane;
            const float *kr, *vr;
            const bool have = pos < kend && rows_of.row(rd.slot, pos, kvh, kr, vr, a.err);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                vreg[i] = have ? __ldg(reinterpret_cast<const float4 *>(vr) + wq + 4 * i)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        auto store_k = [&]() {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float4 h, l;
                split4(kreg[i], h, l);
                const uint32_t off = (lane >> 3) * 8192u + sw128_chunk(warp * 8 + i, lane & 7);
                *reinterpret_cast<float4 *>(Khi + off) = h;
                *reinterpret_cast<float4 *>(Klo + off) = l;
            }
        };
        auto store_v = [&]() {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d0 = 4 * (wq + 4 * i);
                const float v4[4] = {vreg[i].x, vreg[i].y, vreg[i].z, vreg[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float h, l;
                    split_tf32(v4[e], h, l);
                    const uint32_t off = half * 16384u + sw128_offset(d0 + e, lane);
                    *reinterpret_cast<float *>(Vhi + off) = h;
                    *reinterpret_cast<float *>(Vlo + off) = l;
                }
            }
        };
        // MMA issue: after the operand barrier, lane 0 of warp 0 issues QK (and
        // commits it to bar_qk) while lane 0 of warp 4 issues PV (bar_pv); each
        // commit tracks only its own thread's MMAs.
        const uint64_t dKhi = desc_sw128(smem_u32(Khi)), dKlo = desc_sw128(smem_u32(Klo));
        const uint64_t dQlo = desc_sw128(smem_u32(Qlo));
        const uint64_t dVhi = desc_sw128(smem_u32(Vhi)), dVlo = desc_sw128(smem_u32(Vlo));
        auto issue_qk = [&]() {
            const uint32_t tS = tbase + kColS, tQ = tbase + kColQhi;
            const uint32_t idesc_s = idesc_tf32(128, kKT);
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const uint64_t ko = ((s >> 2) * 8192u + (s & 3) * 32u) >> 4;
                const uint64_t qo = ((s >> 2) * 16384u + (s & 3) * 32u) >> 4;
                mma_tf32_ts(tS, tQ + 8 * s, dKhi + ko, idesc_s, s > 0);
                mma_tf32_ts(tS, tQ + 8 * s, dKlo + ko, idesc_s, 1);
                mma_tf32(tS, dQlo + qo, dKhi + ko, idesc_s, 1);
            }
            mma_commit(smem_u32(&bar_qk));
        };
        auto issue_pv = [&](bool first) {
            const uint32_t tD = tbase + kColD, tPh = tbase + kColPhi, tPl = tbase + kColPlo;
            const uint32_t idesc_o = idesc_tf32(128, kHD);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t vo = ((s >> 2) * 16384u + (s & 3) * 32u) >> 4;
                mma_tf32_ts(tD, tPh + 8 * s, dVhi + vo, idesc_o, !first || s > 0);
                mma_tf32_ts(tD, tPh + 8 * s, dVlo + vo, idesc_o, 1);
                mma_tf32_ts(tD, tPl + 8 * s, dVhi + vo, idesc_o, 1);
            }
            mma_commit(smem_u32(&bar_pv));
        };
        auto operands_ready = [&](bool qk, bool pv, bool pv_first) {
            tmem_st_wait();
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
            if (qk && tid == 0) issue_qk();
            if (pv && tid == 128) issue_pv(pv_first);
        };

        // The output accumulator lives in TMEM (D) and the P.V MMAs add into it.
        // p is taken relative to a reference max m_ref that moves only when a
        // tile's max exceeds it by more than kRescale (base-2 units); then D and
        // l are rescaled once.  Both threads of a row take the same decisions.
        float m_ref = -INFINITY, l_run = 0.f;
        uint32_t ph_qk = 0, ph_pv = 0;

        // prologue: K of the first tile; V of the first tile and K of the second in registers
        prefetch_k(kt0);
        prefetch_v(kt0);
        store_k();
        if (kt0 + 1 < kt1) prefetch_k(kt0 + 1);
        operands_ready(kt0 < kt1, false, false);

        for (int kt = kt0; kt < kt1; ++kt) {
            ok = __syncthreads_and(mbar_wait(smem_u32(&bar_qk), ph_qk));
            ph_qk ^= 1;
            if (!ok) break;
            fence_after_sync();

            // this thread's 32 scores; row max and sum shared with the partner
            // thread of the same row (tid ^ 128)
            float s[32];
            tmem_ld32(tbase + tlane + kColS + 32 * half, s);
            const int base = kt * kKT + 32 * half;
            float tmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const bool vis = base + i < kend_row && base + i < kend;
                s[i] = vis ? s[i] : -INFINITY;
                tmax = fmaxf(tmax, s[i]);
            }
            red[0][tid] = tmax;
            __syncthreads();
            const float row_max = fmaxf(tmax, red[0][tid ^ 128]);
            const bool rescale = m_ref != -INFINITY && row_max > m_ref + kRescale;
            const float m_use = (m_ref == -INFINITY || rescale) ? row_max : m_ref;
            float psum = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                s[i] = (s[i] == -INFINITY) ? 0.f : exp2f(s[i] - m_use);
                psum += s[i];
            }
            red[1][tid] = psum;
            __syncthreads();
            const float rowsum = half ? red[1][tid ^ 128] + psum : psum + red[1][tid ^ 128];

            // PV(kt-1) complete: D is quiescent (rescale it if the reference moved)
            if (kt > kt0) {
                ok = __syncthreads_and(mbar_wait(smem_u32(&bar_pv), ph_pv));
                ph_pv ^= 1;
                if (!ok) break;
                fence_after_sync();
            }
            // tcgen05.ld / st are warp-collective: the whole warp takes this branch
            // when any of its rows rescales (the others multiply by 1)
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? exp2f(m_ref - m_use) : 1.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float dv[32];
                    tmem_ld32(tbase + tlane + kColD + 64 * half + 32 * c, dv);
#pragma unroll
                    for (int i = 0; i < 32; ++i) dv[i] *= f;
                    tmem_st32(tbase + tlane + kColD + 64 * half + 32 * c, dv);
                    tmem_st_wait();
                }
                l_run *= f;
            }
            l_run += rowsum;
            m_ref = m_use;

            // P_kt -> TMEM (hi, then lo), V_kt -> smem, K_{kt+1} -> smem
            {
                float t[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = __uint_as_float(__float_as_uint(s[i]) & 0xFFFFE000u);
                tmem_st32(tbase + tlane + kColPhi + 32 * half, t);
                tmem_st_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = s[i] - __uint_as_float(__float_as_uint(s[i]) & 0xFFFFE000u);
                tmem_st32(tbase + tlane + kColPlo + 32 * half, t);
            }
            store_v();
            if (kt + 1 < kt1) {
                store_k();
                prefetch_v(kt + 1);
                if (kt + 2 < kt1) prefetch_k(kt + 2);
            }
            operands_ready(kt + 1 < kt1, true, kt == kt0);
        }
        // the last PV, then the result
        if (ok) ok = __syncthreads_and(mbar_wait(smem_u32(&bar_pv), ph_pv));
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
                      static_cast<size_t>(h) * kHD + 64 * half;
            } else {
                const int n_split = (kend_tile + a.split_keys - 1) / a.split_keys;
                ph = static_cast<size_t>(tile.part0 + (valid ? tq : 0) * n_split + tile.split) * a.n_heads + h;
                dst = a.pacc + ph * kHD + 64 * half;
            }
            const float scl = direct ? 1.f / l_run : 1.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float dv[32];
                tmem_ld32(tbase + tlane + kColD + 64 * half + 32 * c, dv);
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + 32 * c + i) =
                            make_float4(dv[i] * scl, dv[i + 1] * scl, dv[i + 2] * scl, dv[i + 3] * scl);
                }
            }
            if (valid && !direct && half == 0) {
                a.pm[ph] = m_ref;
                a.pl[ph] = l_run;
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

template <int G, class Rows>
cudaError_t launch_prefill_g(const PrefillArgs &a, const Rows &r, cudaStream_t s) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<G, Rows>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const long long grid = static_cast<long long>(a.n_tiles) * a.n_kv;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prefill_tc_kernel<G, Rows><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, s>>>(a, r);
    return cudaGetLastError();
}

template <class Rows>
cudaError_t launch_prefill(const PrefillArgs &a, const Rows &r, cudaStream_t s) {
    switch (a.group) {
        case 1: return launch_prefill_g<1>(a, r, s);
        case 2: return launch_prefill_g<2>(a, r, s);
        case 4: return launch_prefill_g<4>(a, r, s);
        case 8: return launch_prefill_g<8>(a, r, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill_paged(const PrefillArgs &a, const PagedAddr &addr, cudaStream_t s) {
    return launch_prefill(a, PagedRowsP{addr}, s);
}

cudaError_t launch_prefill_contig(const PrefillArgs &a, const ContigAddr &addr, cudaStream_t s) {
    return launch_prefill(a, ContigRowsP{addr}, s);
}

}  // namespace pkv
