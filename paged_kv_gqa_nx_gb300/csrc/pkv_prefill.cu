// pkv_prefill.cu -- tensor-core attention for chunked-prefill rows (n_q > 1).
//
// For a row with many new tokens, Q.K^T over a tile of queries and keys is a
// real dense contraction, so it runs on the 5th-generation tensor cores
// (tcgen05.mma kind::tf32).  To keep f32 accuracy each f32 operand x is split
// into a tf32 part and its exact f32 rest (x = hi + lo) and every product is
// formed as hi*hi + hi*lo + lo*hi; the dropped lo*lo term is ~2^-20 relative.
//
// One CTA (128 threads) = one tile of 128 query rows -- (128 / G) consecutive
// tokens x the G query heads that share kv head `kvh` -- and one key split.
// Row m of the tile is token m / G, head m % G, and TMEM lane m; thread m owns
// that row's online softmax.  Per key tile of 32 positions:
//   1. K and V rows (through the page table or a contiguous history) are
//      split into hi/lo and written to shared memory as the K-major B operand
//      of Q.K^T and, transposed, of P.V;
//   2. S[128 x 32] = Q.K^T into TMEM (48 MMAs of K = 8);
//   3. each thread reads its row of S, applies the offset-causal mask
//      (key j visible iff j <= q_pos = total_k - n_q + i), updates (max, sum)
//      and writes p (hi/lo) as the A operand of P.V;
//   4. D[128 x 128] = P.V into TMEM (12 MMAs); each thread adds its row of D
//      to its register accumulator after rescaling.
// The next tile's K/V rows are loaded into registers while the MMAs run.
// Shared memory: Q hi/lo 128 KiB, K hi/lo (aliased by P hi/lo) 32 KiB, V^T
// hi/lo 32 KiB.  TMEM: 256 columns (D at 0, S at 128).
//
// The address functor is the decode kernels' (PagedRows / ContigRows), so the
// paged and contiguous instantiations return the same bits.
#include "pkv_internal.h"
#include "pkv_tcgen05.h"

namespace pkv {
namespace {

using namespace tc;

constexpr int kHD = 128;
constexpr int kKT = 32;          // keys per tile
constexpr uint32_t kTmemCols = 256;

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
};

constexpr size_t kSmemQ = 64 * 1024;       // one of Q hi / Q lo
constexpr size_t kSmemK = 16 * 1024;       // one of K hi / K lo (and P hi / P lo)
constexpr size_t kSmemV = 16 * 1024;       // one of V^T hi / V^T lo
constexpr size_t kSmemBytes = 2 * kSmemQ + 2 * kSmemK + 2 * kSmemV + 1024;  // + alignment slack

__device__ __forceinline__ void split4(const float4 &x, float4 &h, float4 &l) {
    split_tf32(x.x, h.x, l.x);
    split_tf32(x.y, h.y, l.y);
    split_tf32(x.z, h.z, l.z);
    split_tf32(x.w, h.w, l.w);
}

template <int G, class Rows>
__global__ void __launch_bounds__(128, 1) prefill_tc_kernel(PrefillArgs a, Rows rows_of) {
    constexpr int TQ = 128 / G;  // tokens per tile
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *Qhi = sm;
    unsigned char *Qlo = Qhi + kSmemQ;
    unsigned char *Khi = Qlo + kSmemQ;   // also P hi
    unsigned char *Klo = Khi + kSmemK;   // also P lo
    unsigned char *Vhi = Klo + kSmemK;
    unsigned char *Vlo = Vhi + kSmemV;
    __shared__ uint64_t mbar;
    __shared__ uint32_t tslot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ti = blockIdx.x / a.n_kv;
    const int kvh = blockIdx.x - ti * a.n_kv;
    const PrefillTile tile = a.tiles[ti];
    const RowDesc rd = a.rows[tile.row];
    const int total_k = rd.past_len + rd.n_q;

    // this thread's row of the tile
    const int tq = tid / G, g = tid - (tid / G) * G;
    const int qi = tile.q0 + tq;
    const bool valid = qi < rd.n_q;
    const int q_pos = total_k - rd.n_q + qi;
    const int kend_row = valid ? (a.causal ? min(q_pos + 1, total_k) : total_k) : 1;

    // key range of this split
    const int n_valid_q = min(TQ, rd.n_q - tile.q0);
    const int kend_tile =
        a.causal ? min(total_k, total_k - rd.n_q + tile.q0 + n_valid_q) : total_k;
    const int kbeg = tile.split * a.split_keys;
    const int kend = min(kbeg + a.split_keys, kend_tile);
    const int kt0 = kbeg / kKT, kt1 = (kend + kKT - 1) / kKT;

    // Q row (pre-scaled to base-2 units), split into the A operand
    {
        const float *qrow = a.Q + static_cast<size_t>(rd.q_row0 + (valid ? qi : 0)) * (a.n_heads * kHD) +
                            static_cast<size_t>(kvh * G + g) * kHD;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            float4 x = valid ? __ldg(reinterpret_cast<const float4 *>(qrow) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            x.x *= a.scale_log2;
            x.y *= a.scale_log2;
            x.z *= a.scale_log2;
            x.w *= a.scale_log2;
            float4 h, l;
            split4(x, h, l);
            const uint32_t off = (j >> 3) * 16384u + sw128_chunk(tid, j & 7);
            *reinterpret_cast<float4 *>(Qhi + off) = h;
            *reinterpret_cast<float4 *>(Qlo + off) = l;
        }
    }
    if (tid == 0) mbar_init(smem_u32(&mbar), 1);
    if (warp == 0) {
        tmem_alloc(smem_u32(&tslot), kTmemCols);
        tmem_relinquish();
    }

    // register prefetch of one key tile: K rows key-major (8 keys per warp,
    // one 512-byte row per instruction), V rows key-per-lane (for the transpose)
    float4 kreg[8], vreg[8];
    auto prefetch = [&](int kt) {
        const int base = kt * kKT;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int pos = base + warp * 8 + i;
            kreg[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            const float *kr, *vr;
            if (pos < kend && rows_of.row(rd.slot, pos, kvh, kr, vr, a.err))
                kreg[i] = __ldg(reinterpret_cast<const float4 *>(kr) + lane);
        }
        const int vpos = base + lane;
        const float *kr, *vr;
        const bool vok = vpos < kend && rows_of.row(rd.slot, vpos, kvh, kr, vr, a.err);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            vreg[i] = vok ? __ldg(reinterpret_cast<const float4 *>(vr) + warp + 4 * i)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if (kt0 < kt1) prefetch(kt0);

    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;
    const uint32_t tlane = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t tS = tbase + 128, tD = tbase;
    const uint32_t idesc_s = idesc_tf32(128, kKT), idesc_o = idesc_tf32(128, kHD);

    float o[kHD];
#pragma unroll
    for (int d = 0; d < kHD; ++d) o[d] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t phase = 0;
    bool ok = true;

    for (int kt = kt0; kt < kt1 && ok; ++kt) {
        // 1. K (B operand of Q.K^T) and V^T (B operand of P.V), hi and lo
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int key = warp * 8 + i;
            float4 h, l;
            split4(kreg[i], h, l);
            const uint32_t off = (lane >> 3) * 4096u + sw128_chunk(key, lane & 7);
            *reinterpret_cast<float4 *>(Khi + off) = h;
            *reinterpret_cast<float4 *>(Klo + off) = l;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int d0 = 4 * (warp + 4 * i);
            const float v4[4] = {vreg[i].x, vreg[i].y, vreg[i].z, vreg[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float h, l;
                split_tf32(v4[e], h, l);
                const uint32_t off = sw128_offset(d0 + e, lane);
                *reinterpret_cast<float *>(Vhi + off) = h;
                *reinterpret_cast<float *>(Vlo + off) = l;
            }
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // 2. S = Q.K^T
        if (tid == 0) {
#pragma unroll 1
            for (int s = 0; s < 16; ++s) {
                const uint32_t ao = (s >> 2) * 16384u + (s & 3) * 32u;
                const uint32_t bo = (s >> 2) * 4096u + (s & 3) * 32u;
                const uint64_t qh = desc_sw128(smem_u32(Qhi + ao)), ql = desc_sw128(smem_u32(Qlo + ao));
                const uint64_t kh = desc_sw128(smem_u32(Khi + bo)), kl = desc_sw128(smem_u32(Klo + bo));
                mma_tf32(tS, qh, kh, idesc_s, s > 0);
                mma_tf32(tS, qh, kl, idesc_s, 1);
                mma_tf32(tS, ql, kh, idesc_s, 1);
            }
            mma_commit(smem_u32(&mbar));
        }
        if (kt + 1 < kt1) prefetch(kt + 1);
        ok = __syncthreads_and(mbar_wait(smem_u32(&mbar), phase));
        phase ^= 1;
        if (!ok) break;
        fence_after_sync();

        // 3. online softmax of this row over the tile's 32 keys
        float s[32];
        tmem_ld32(tS + tlane, s);
        const int base = kt * kKT;
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const bool vis = base + i < kend_row && base + i < kend;
            s[i] = vis ? s[i] : -INFINITY;
            tmax = fmaxf(tmax, s[i]);
        }
        const float m_new = fmaxf(m_run, tmax);
        const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            s[i] = (s[i] == -INFINITY) ? 0.f : exp2f(s[i] - m_new);
            psum += s[i];
        }
        l_run = fmaf(l_run, alpha, psum);
        m_run = m_new;
        // p (A operand of P.V) over the K hi/lo space, row tid
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float4 p = make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
            float4 h, l;
            split4(p, h, l);
            const uint32_t off = sw128_chunk(tid, c);
            *reinterpret_cast<float4 *>(Khi + off) = h;
            *reinterpret_cast<float4 *>(Klo + off) = l;
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();

        // 4. D = P.V
        if (tid == 0) {
#pragma unroll 1
            for (int st = 0; st < 4; ++st) {
                const uint32_t off = st * 32u;
                const uint64_t ph = desc_sw128(smem_u32(Khi + off)), pl = desc_sw128(smem_u32(Klo + off));
                const uint64_t vh = desc_sw128(smem_u32(Vhi + off)), vl = desc_sw128(smem_u32(Vlo + off));
                mma_tf32(tD, ph, vh, idesc_o, st > 0);
                mma_tf32(tD, ph, vl, idesc_o, 1);
                mma_tf32(tD, pl, vh, idesc_o, 1);
            }
            mma_commit(smem_u32(&mbar));
        }
        ok = __syncthreads_and(mbar_wait(smem_u32(&mbar), phase));
        phase ^= 1;
        if (!ok) break;
        fence_after_sync();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float dv[32];
            tmem_ld32(tD + tlane + 32 * c, dv);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[32 * c + i] = fmaf(o[32 * c + i], alpha, dv[i]);
        }
        fence_before_sync();
        __syncthreads();
    }

    if (!ok) {
        if (tid == 0 && a.err) atomicOr(a.err, 2);
    } else if (valid) {
        const int h = kvh * G + g;
        if (tile.part0 < 0) {
            float *orow = a.out + static_cast<size_t>(rd.q_row0 + qi) * (a.n_heads * kHD) +
                          static_cast<size_t>(h) * kHD;
            const float inv = 1.f / l_run;
#pragma unroll
            for (int d = 0; d < kHD; d += 4)
                *reinterpret_cast<float4 *>(orow + d) =
                    make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
        } else {
            const int n_split = (kend_tile + a.split_keys - 1) / a.split_keys;
            const size_t ph = static_cast<size_t>(tile.part0 + tq * n_split + tile.split) * a.n_heads + h;
            float *prow = a.pacc + ph * kHD;
#pragma unroll
            for (int d = 0; d < kHD; d += 4)
                *reinterpret_cast<float4 *>(prow + d) = make_float4(o[d], o[d + 1], o[d + 2], o[d + 3]);
            a.pm[ph] = m_run;
            a.pl[ph] = l_run;
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
    prefill_tc_kernel<G, Rows><<<static_cast<unsigned>(grid), 128, kSmemBytes, s>>>(a, r);
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
