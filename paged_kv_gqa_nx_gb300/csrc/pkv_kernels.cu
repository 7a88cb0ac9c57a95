// pkv_kernels.cu -- sm_103a kernels of libpkv.
//
//   prep          one launch per layer call: upload changed page-table entries
//                 and scatter the layer's K_new / V_new rows into their blocks
//                 (the append step of "nx_f32_attn_paged.nx source")
//   pt_apply      page-table upload alone (pkv_pool_flush)
//   copy_blocks   copy-on-append: duplicate shared blocks (every layer, K and V)
//   decode_fast   split-K attention, head_dim 128, query group 1/2/4: one CTA
//                 per (work unit, kv head); the whole GQA group of query heads
//                 reuses every K/V row ("nx_f32_attn_paged.nx source", step 3:
//                 query head h reads kv head h / group)
//   decode_generic the same computation for any head_dim <= 256 and group
//   merge_splits  log-sum-exp merge of the split partials
//
// The attention kernels are templates over an address functor: PagedAddr
// reads rows through the page table (f32 or bf16 pool elements, widened to
// f32 on load), ContigAddr from a contiguous f32 history.
// Everything else -- the split boundaries (multiples of S keys), the tile
// order, every reduction tree -- depends only on token positions, so the paged
// and the contiguous instantiations return the same bits, and a batch row
// returns the same bits as the same row launched alone.
#include "pkv_elem.h"
#include "pkv_internal.h"
#include "pkv_rows.h"

#include <cstdio>
#include <type_traits>

namespace pkv {
namespace {

// ------------------------------------------------------------- page table ----

__global__ void pt_apply_kernel(int32_t *pt, int32_t max_blocks, const PtRun *runs,
                                const int32_t *vals) {
    const PtRun r = runs[blockIdx.x];
    int32_t *dst = pt + static_cast<size_t>(r.slot) * max_blocks + r.start;
    for (int i = threadIdx.x; i < r.count; i += blockDim.x) dst[i] = vals[r.voff + i];
}

// ----------------------------------------------------------------- append ----


// ------------------------------------------------------------------- prep ----
//
// One launch before attention: blocks [0, n_runs) upload page-table runs, the
// other blocks append the new rows (8 warps per block, one warp per row and K
// or V; the destination block comes from the host's page table).

// RoPE (NeoX pairing) of one appended row, all heads: K into its pool row,
// or Q into Q_rot.  Lane l takes the pairs (i, i + hd/2) for i = l, l + 32,
// ..., the angle pos * base^(-2i/hd) and its cosine and sine computed in
// double precision and rounded to f32 once; the rotation is f32.
__device__ void rope_row(const PrepArgs &p, const PagedAddr &a, const AppendDesc &d, bool is_q,
                         int lane) {
    const int half = p.hd >> 1;
    const float *src;
    float *dst = nullptr;       // the rotated queries
    size_t dst_off = 0;         // or the key row in the pool (f32 or bf16 elements)
    int n_heads;
    if (is_q) {
        src = p.Q + static_cast<size_t>(d.src_row) * p.q_dim;
        dst = p.Q_rot + static_cast<size_t>(d.src_row) * p.q_dim;
        n_heads = p.q_dim / p.hd;
    } else {
        if (static_cast<unsigned>(d.blk) >= static_cast<unsigned>(a.n_blocks)) {
            if (lane == 0) flag_error(p.err, 1);
            return;
        }
        const int off = a.bs_shift >= 0 ? (d.pos & (a.bs - 1)) : (d.pos % a.bs);
        src = p.K_new + static_cast<size_t>(d.src_row) * a.kv_dim;
        dst_off = static_cast<size_t>(d.blk) * a.block_stride + a.layer_off +
                  static_cast<size_t>(off) * a.kv_dim;
        n_heads = a.kv_dim / p.hd;
    }
    const double lb = log(p.rope_base);
    for (int i = lane; i < half; i += 32) {
        const double ang = static_cast<double>(d.pos) * exp(-2.0 * i / p.hd * lb);
        double sd, cd;
        sincos(ang, &sd, &cd);
        const float c = static_cast<float>(cd), sn = static_cast<float>(sd);
        for (int h = 0; h < n_heads; ++h) {
            const float x0 = src[h * p.hd + i], x1 = src[h * p.hd + i + half];
            // products and sums each rounded to f32 (no contraction), so the
            // value that a bf16 pool rounds is reproducible
            const float y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
            const float y1 = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
            const size_t o0 = static_cast<size_t>(h) * p.hd + i, o1 = o0 + half;
            if (dst) {
                dst[o0] = y0;
                dst[o1] = y1;
            } else if (a.fp8) {
                const float inv = 1.f / a.kv_scale;
                store1(static_cast<fp8 *>(a.k) + dst_off + o0, y0 * inv);
                store1(static_cast<fp8 *>(a.k) + dst_off + o1, y1 * inv);
            } else if (a.bf16) {
                store1(static_cast<bf16 *>(a.k) + dst_off + o0, y0);
                store1(static_cast<bf16 *>(a.k) + dst_off + o1, y1);
            } else {
                store1(static_cast<float *>(a.k) + dst_off + o0, y0);
                store1(static_cast<float *>(a.k) + dst_off + o1, y1);
            }
        }
    }
}

__global__ void prep_kernel(PrepArgs p, PagedAddr a) {
    int b = blockIdx.x;
    if (b < p.n_runs) {
        const PtRun r = p.runs[b];
        int32_t *dst = p.pt + static_cast<size_t>(r.slot) * p.max_blocks + r.start;
        for (int i = threadIdx.x; i < r.count; i += blockDim.x) dst[i] = p.vals[r.voff + i];
        return;
    }
    b -= p.n_runs;
    const bool rope = p.rope_base > 0.0;
    const int per_row = rope ? 3 : 2;  // warps per appended row: K, V (, Q)
    const int app_blocks = (per_row * p.n_app + 7) / 8;
    if (b < app_blocks) {
        const int gw = b * 8 + (threadIdx.x >> 5);
        const int lane = threadIdx.x & 31;
        if (gw >= per_row * p.n_app) return;
        const AppendDesc d = p.app[gw / per_row];
        const int role = gw - (gw / per_row) * per_row;  // 0 K, 1 V, 2 Q
        if (rope && role != 1) {
            rope_row(p, a, d, role == 2, lane);
            return;
        }
        const bool is_v = role == 1;
        if (static_cast<unsigned>(d.blk) >= static_cast<unsigned>(a.n_blocks)) {
            if (lane == 0) flag_error(p.err, 1);
            return;
        }
        const int off = a.bs_shift >= 0 ? (d.pos & (a.bs - 1)) : (d.pos % a.bs);
        const size_t o = static_cast<size_t>(d.blk) * a.block_stride + a.layer_off +
                         static_cast<size_t>(off) * a.kv_dim;
        const float *src = (is_v ? p.V_new : p.K_new) + static_cast<size_t>(d.src_row) * a.kv_dim;
        void *base = is_v ? a.v : a.k;
        if (a.fp8) {
            fp8 *dst = static_cast<fp8 *>(base) + o;
            const float inv = 1.f / a.kv_scale;  // power of two: exact
            if (p.vec4)
                for (int i = lane; i < (a.kv_dim >> 2); i += 32) {
                    const float4 x = ldg4(src + 4 * i);
                    store4(dst + 4 * i, make_float4(x.x * inv, x.y * inv, x.z * inv, x.w * inv));
                }
            else
                for (int i = lane; i < a.kv_dim; i += 32) store1(dst + i, src[i] * inv);
        } else if (a.bf16) {
            bf16 *dst = static_cast<bf16 *>(base) + o;
            if (p.vec4)
                for (int i = lane; i < (a.kv_dim >> 2); i += 32) store4(dst + 4 * i, ldg4(src + 4 * i));
            else
                for (int i = lane; i < a.kv_dim; i += 32) store1(dst + i, src[i]);
        } else {
            float *dst = static_cast<float *>(base) + o;
            if (p.vec4)
                for (int i = lane; i < (a.kv_dim >> 2); i += 32) store4(dst + 4 * i, ldg4(src + 4 * i));
            else
                for (int i = lane; i < a.kv_dim; i += 32) dst[i] = src[i];
        }
    }
}

// ------------------------------------------------------------- block copy ----

// Blocks are copied as 4-byte words (block_floats = the block's size in words).
__global__ void copy_blocks_kernel(float *k, float *v, const CopyDesc *__restrict__ items,
                                   int64_t block_floats, int32_t n_blocks, int32_t *err) {
    const CopyDesc c = items[blockIdx.y];
    if (static_cast<unsigned>(c.src) >= static_cast<unsigned>(n_blocks) ||
        static_cast<unsigned>(c.dst) >= static_cast<unsigned>(n_blocks)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(err, 1);
        return;
    }
    const size_t so = static_cast<size_t>(c.src) * block_floats;
    const size_t dO = static_cast<size_t>(c.dst) * block_floats;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    if ((block_floats & 3) == 0) {
        const size_t n4 = static_cast<size_t>(block_floats) >> 2;
        const float4 *ks = reinterpret_cast<const float4 *>(k + so);
        const float4 *vs = reinterpret_cast<const float4 *>(v + so);
        float4 *kd = reinterpret_cast<float4 *>(k + dO);
        float4 *vd = reinterpret_cast<float4 *>(v + dO);
        for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
            kd[i] = ks[i];
            vd[i] = vs[i];
        }
    } else {
        for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < static_cast<size_t>(block_floats);
             i += stride) {
            k[dO + i] = k[so + i];
            v[dO + i] = v[so + i];
        }
    }
}

// ------------------------------------------------- fast decode, hd = 128 ----
//
// CTA = 4 warps = one (unit, kv head).  The unit's keys are cut into tiles of
// T = 8 positions; warp w takes tiles w, w+4, w+8, ... and runs its own
// NST-stage cp.async pipeline and its own online softmax over them (no block
// barrier in the main loop).  The four warps' (max, sum, acc) are combined at
// the end in warp order.
//
// Lane layout for Q.K: lane = 8*kg + c.  Lane group kg handles key kg (and
// kg + 4) of a tile; lane c holds dims {4c + 32i + e : i < 4, e < 4} of every
// query head of the group (16 dims x G heads, pre-scaled by scale*log2(e)).
// The 8 lanes of a group reduce their G partial dot products with a
// reduce-scatter butterfly (xor 4, 2, 1); afterwards lane c holds the full
// score of head c / (8 / G).  Lane layout for P.V: lane owns dims
// 4*lane .. 4*lane+3 of every head.

template <int G, class E = float>
struct FastCfg {
    static constexpr int HD = 128;
    // keys per tile: 8 for f32 rows; 16 for bf16 / fp8 rows, whose smaller
    // stages leave room to spread each tile's softmax over twice the keys
    static constexpr int T = sizeof(E) == 4 ? 8 : 16;
    static constexpr int NIT = T / 4;  // keys per lane group and tile
    static constexpr int W = 4;   // warps per CTA
    static constexpr int LPH = 8 / G;  // lanes of a group holding one head's score
};

template <int G>
__device__ __forceinline__ float reduce_scatter8(const float (&p)[G], int c);

template <>
__device__ __forceinline__ float reduce_scatter8<4>(const float (&p)[4], int c) {
    const bool hi4 = (c & 4) != 0;
    const float s0 = hi4 ? p[0] : p[2], s1 = hi4 ? p[1] : p[3];
    float k0 = hi4 ? p[2] : p[0], k1 = hi4 ? p[3] : p[1];
    k0 += __shfl_xor_sync(kFull, s0, 4);
    k1 += __shfl_xor_sync(kFull, s1, 4);
    const bool hi2 = (c & 2) != 0;
    const float s = hi2 ? k0 : k1;
    float k = hi2 ? k1 : k0;
    k += __shfl_xor_sync(kFull, s, 2);
    k += __shfl_xor_sync(kFull, k, 1);
    return k;  // head c >> 1
}
template <>
__device__ __forceinline__ float reduce_scatter8<2>(const float (&p)[2], int c) {
    const bool hi4 = (c & 4) != 0;
    const float s = hi4 ? p[0] : p[1];
    float k = hi4 ? p[1] : p[0];
    k += __shfl_xor_sync(kFull, s, 4);
    k += __shfl_xor_sync(kFull, k, 2);
    k += __shfl_xor_sync(kFull, k, 1);
    return k;  // head c >> 2
}
template <>
__device__ __forceinline__ float reduce_scatter8<1>(const float (&p)[1], int) {
    float k = p[0];
    k += __shfl_xor_sync(kFull, k, 4);
    k += __shfl_xor_sync(kFull, k, 2);
    k += __shfl_xor_sync(kFull, k, 1);
    return k;
}

__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ float4 fma4(float s, const float4 &v, const float4 &acc) {
    return make_float4(fmaf(s, v.x, acc.x), fmaf(s, v.y, acc.y), fmaf(s, v.z, acc.z),
                       fmaf(s, v.w, acc.w));
}

template <int G, int NST, class E>
constexpr size_t fast_smem_bytes() {
    using C = FastCfg<G, E>;
    return static_cast<size_t>(C::W) * NST * C::T * C::HD * 2 * sizeof(E) +
           static_cast<size_t>(C::W) * (C::T + 1) * 4 * sizeof(float);
}

template <int G, int NST, class Rows>
__global__ void __launch_bounds__(128, 3) decode_fast_kernel(AttnArgs a, Rows rows_of) {
    using E = typename Rows::Elem;             // pool element (f32, bf16 or fp8)
    using C = FastCfg<G, E>;
    constexpr int HD = C::HD, T = C::T, W = C::W, NIT = C::NIT;
    constexpr int EPC = 16 / static_cast<int>(sizeof(E));  // elements per 16-byte chunk
    constexpr int CPR = HD / EPC;              // chunks per row: 32 (f32), 16 (bf16)
    constexpr int STAGE = T * HD * 2;          // elements: K rows then V rows
    constexpr int WARP_ELEMS = NST * STAGE;
    static_assert(NST * STAGE * sizeof(E) >= (G * HD + 2 * G) * sizeof(float),
                  "a warp's stage memory holds its (acc, m, l)");
    extern __shared__ __align__(16) unsigned char smraw[];
    E *sm = reinterpret_cast<E *>(smraw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kg = lane >> 3, c = lane & 7;
    const int ui = blockIdx.x / a.n_kv;
    const int kvh = blockIdx.x - ui * a.n_kv;
    const UnitDesc u = a.units[ui];
    const RowDesc rd = a.rows[u.row];
    const UnitRange ur = unit_range(u, rd, a.causal, a.split_keys);
    const int n_tiles = (ur.kend - ur.kbeg + T - 1) / T;
    const int my_n = warp < n_tiles ? (n_tiles - warp + W - 1) / W : 0;

    E *wbase = sm + warp * WARP_ELEMS;
    float *P = reinterpret_cast<float *>(sm + W * WARP_ELEMS) + warp * (T + 1) * 4;

    // query slice of the group, pre-scaled to base-2 units
    const float *qrow = a.Q + static_cast<size_t>(rd.q_row0 + u.qi) * (a.n_heads * HD) +
                        static_cast<size_t>(kvh) * G * HD;
    // an fp8 pool's power-of-two scale folds into the queries (for K) and the
    // output (for V), exactly; it is 1 on other pools
    const float ks = rows_of.scale();
    float4 q[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 t = __ldg(reinterpret_cast<const float4 *>(qrow + g * HD + 4 * c + 32 * i));
            q[g][i] = make_float4(t.x * a.scale_log2 * ks, t.y * a.scale_log2 * ks,
                                  t.z * a.scale_log2 * ks, t.w * a.scale_log2 * ks);
        }

    const bool whole = rows_of.whole_tiles(T);
    const size_t rstride = rows_of.row_stride();
    // fused append (f32 pools): positions from past_len on come from K_new / V_new
    constexpr bool kF32 = std::is_same<E, float>::value;
    const bool fused = kF32 && a.K_new != nullptr;
    const int new0 = fused ? rd.past_len : 0x7fffffff;
    auto row_ptrs = [&](int pos, const E *&kr, const E *&vr) {
        if constexpr (kF32) {
            if (pos >= new0) {
                const size_t o = static_cast<size_t>(rd.q_row0 + (pos - new0)) * rstride +
                                 static_cast<size_t>(kvh) * HD;
                kr = a.K_new + o;
                vr = a.V_new + o;
                return true;
            }
        }
        return rows_of.row(rd.slot, pos, kvh, HD, kr, vr, a.err);
    };
    // one key's K and V rows into the stage: 2 * CPR 16-byte chunks over the lanes
    auto copy_rows = [&](E *Kd, E *Vd, const E *kr, const E *vr) {
#pragma unroll
        for (int ci = lane; ci < 2 * CPR; ci += 32) {
            if (ci < CPR) cp_async16(Kd + ci * EPC, kr + ci * EPC);
            else cp_async16(Vd + (ci - CPR) * EPC, vr + (ci - CPR) * EPC);
        }
    };
    auto load_tile = [&](int k_local, int stage) {
        const int pos0 = ur.kbeg + (warp + k_local * W) * T;
        const int nv = min(T, ur.kend - pos0);
        E *Ks = wbase + stage * STAGE;
        E *Vs = Ks + T * HD;
        if (whole && pos0 + T <= new0) {
            // one page-table lookup per tile
            const E *kb, *vb;
            if (rows_of.row(rd.slot, pos0, kvh, HD, kb, vb, a.err)) {
#pragma unroll
                for (int j = 0; j < T; ++j)
                    if (j < nv) copy_rows(Ks + j * HD, Vs + j * HD, kb + j * rstride, vb + j * rstride);
            }
        } else {
#pragma unroll
            for (int j = 0; j < T; ++j) {
                if (j < nv) {
                    const E *kr, *vr;
                    if (row_ptrs(pos0 + j, kr, vr)) copy_rows(Ks + j * HD, Vs + j * HD, kr, vr);
                }
            }
        }
    };

#pragma unroll
    for (int s = 0; s < NST - 1; ++s) {
        if (s < my_n) load_tile(s, s);
        cp_async_commit();
    }

    // fused append: the unit of the row's last query stores the new rows of
    // its split into the pool (nothing in this launch reads them from there;
    // the first tiles' copies are already in flight)
    if (kF32 && fused && u.qi == rd.n_q - 1) {
        for (int pos = max(ur.kbeg, new0) + warp; pos < ur.kend; pos += W) {
            const int t = pos - new0;
            const AppendDesc ad = a.app[rd.q_row0 + t];
            const size_t o = static_cast<size_t>(rd.q_row0 + t) * rstride + static_cast<size_t>(kvh) * HD;
            const bool set_pt = a.pt_write && kvh == 0 && (pos == 0 || rows_of.block_start(pos));
            rows_of.store_row(rd.slot, ad.blk, pos, kvh, HD, a.K_new + o, a.V_new + o, set_pt, lane, a.err);
        }
    }

    constexpr int LPH = C::LPH;
    const int hh = c / LPH;  // the head whose score this lane holds
    float m_run = -INFINITY, l_run = 0.f;
    float4 acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int k = 0; k < my_n; ++k) {
        const int kn = k + NST - 1;
        if (kn < my_n) load_tile(kn, kn % NST);
        cp_async_commit();
        cp_async_wait<NST - 1>();
        __syncwarp();

        const int pos0 = ur.kbeg + (warp + k * W) * T;
        const int n_valid = min(T, ur.kend - pos0);
        const E *Ks = wbase + (k % NST) * STAGE;
        const E *Vs = Ks + T * HD;

        float sc[NIT];
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int j = it * 4 + kg;
            float4 kk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) kk[i] = load4(Ks + j * HD + 4 * (c + 8 * i));
            float part[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float acc_d = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc_d = fmaf(q[g][i].x, kk[i].x, acc_d);
                    acc_d = fmaf(q[g][i].y, kk[i].y, acc_d);
                    acc_d = fmaf(q[g][i].z, kk[i].z, acc_d);
                    acc_d = fmaf(q[g][i].w, kk[i].w, acc_d);
                }
                part[g] = acc_d;
            }
            const float s = reduce_scatter8<G>(part, c);
            sc[it] = (j < n_valid) ? s : -INFINITY;
        }

        // online softmax for this lane's head over the tile's T keys
        float tmax = fmaxf(sc[0], sc[1]);
#pragma unroll
        for (int it = 2; it < NIT; ++it) tmax = fmaxf(tmax, sc[it]);
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
        const float m_new = fmaxf(m_run, tmax);
        const float alpha = exp2f(m_run - m_new);
        float pv[NIT];
#pragma unroll
        for (int it = 0; it < NIT; ++it) pv[it] = exp2f(sc[it] - m_new);
        float ps = pv[0] + pv[1];
#pragma unroll
        for (int it = 2; it < NIT; ++it) ps += pv[it];
        ps += __shfl_xor_sync(kFull, ps, 8);
        ps += __shfl_xor_sync(kFull, ps, 16);
        l_run = fmaf(l_run, alpha, ps);
        m_run = m_new;
        if ((c % LPH) == 0) {
#pragma unroll
            for (int it = 0; it < NIT; ++it) P[(it * 4 + kg) * 4 + hh] = pv[it];
            if (kg == 0) P[T * 4 + hh] = alpha;
        }
        __syncwarp();

        const float4 *P4 = reinterpret_cast<const float4 *>(P);
        const float4 al = P4[T];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float s = comp(al, g);
            acc[g] = make_float4(acc[g].x * s, acc[g].y * s, acc[g].z * s, acc[g].w * s);
        }
#pragma unroll
        for (int j = 0; j < T; ++j) {
            if (j < n_valid) {
                const float4 v = load4(Vs + j * HD + 4 * lane);
                const float4 pj = P4[j];
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = fma4(comp(pj, g), v, acc[g]);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncwarp();

    // publish this warp's state in its own (now idle) stage memory
    float *R = reinterpret_cast<float *>(wbase);
    auto Rw = [&](int w) { return reinterpret_cast<const float *>(sm + w * WARP_ELEMS); };
#pragma unroll
    for (int g = 0; g < G; ++g) reinterpret_cast<float4 *>(R + g * HD)[lane] = acc[g];
    if (kg == 0 && (c % LPH) == 0) {
        R[G * HD + hh] = m_run;
        R[G * HD + G + hh] = l_run;
    }
    __syncthreads();

    const int d = threadIdx.x;  // 128 threads <-> 128 dims
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float mw[W];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            mw[w] = Rw(w)[G * HD + g];
            M = fmaxf(M, mw[w]);
        }
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            if (mw[w] != -INFINITY) {
                const float wt = exp2f(mw[w] - M);
                num = fmaf(wt, Rw(w)[g * HD + d], num);
                den = fmaf(wt, Rw(w)[G * HD + G + g], den);
            }
        }
        const int h = kvh * G + g;
        if (u.item < 0) {
            a.out[static_cast<size_t>(rd.q_row0 + u.qi) * (a.n_heads * HD) +
                  static_cast<size_t>(h) * HD + d] = num * ks / den;
        } else {
            const size_t ph = static_cast<size_t>(a.merges[u.item].part0 + u.split) * a.n_heads + h;
            a.pacc[ph * HD + d] = num * ks;
            if (d == 0) {
                a.pm[ph] = M;
                a.pl[ph] = den;
            }
        }
    }
}

// --------------------------------------------------------- generic decode ----
//
// CTA = 4 warps = one (unit, kv head, chunk of up to 16 query heads).  Warp w
// takes the unit's keys w, w+4, ...; for each key and head the warp forms the
// dot product over lanes (d = lane, lane+32, ...) and a butterfly sum, then
// updates its online softmax; the accumulators live in shared memory.

constexpr int kGenW = 4;
constexpr int kGenMaxHeads = 16;

__host__ __device__ constexpr size_t generic_smem_floats(int hpc, int hd) {
    return static_cast<size_t>(hpc) * hd * (1 + kGenW) + 2 * kGenW * hpc;
}

template <class Rows>
__global__ void __launch_bounds__(128) decode_generic_kernel(AttnArgs a, Rows rows_of, int hpc) {
    extern __shared__ __align__(16) float sm[];
    const int n_chunks = (a.group + hpc - 1) / hpc;
    int b = blockIdx.x;
    const int chunk = b % n_chunks;
    b /= n_chunks;
    const int kvh = b % a.n_kv;
    const int ui = b / a.n_kv;
    const UnitDesc u = a.units[ui];
    const RowDesc rd = a.rows[u.row];
    const UnitRange ur = unit_range(u, rd, a.causal, a.split_keys);
    const int hd = a.hd;
    const int h0 = kvh * a.group + chunk * hpc;
    const int nh = min(hpc, a.group - chunk * hpc);

    float *qs = sm;                                // [hpc][hd]
    float *accs = qs + hpc * hd;                   // [W][hpc][hd]
    float *ms = accs + kGenW * hpc * hd;           // [W][hpc]
    float *ls = ms + kGenW * hpc;                  // [W][hpc]
    const float *qrow = a.Q + static_cast<size_t>(rd.q_row0 + u.qi) * (a.n_heads * hd) +
                        static_cast<size_t>(h0) * hd;
    const float ks = rows_of.scale();  // fp8 scale (power of two) into the queries and the output
    for (int t = threadIdx.x; t < nh * hd; t += blockDim.x) qs[t] = qrow[t] * a.scale_log2 * ks;
    for (int t = threadIdx.x; t < kGenW * hpc * hd; t += blockDim.x) accs[t] = 0.f;
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float m[kGenMaxHeads], l[kGenMaxHeads];
#pragma unroll
    for (int g = 0; g < kGenMaxHeads; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
    }
    float *acc = accs + warp * hpc * hd;
    for (int j = ur.kbeg + warp; j < ur.kend; j += kGenW) {
        const typename Rows::Elem *kr, *vr;
        if (!rows_of.row(rd.slot, j, kvh, hd, kr, vr, a.err)) continue;
#pragma unroll
        for (int g = 0; g < kGenMaxHeads; ++g) {
            if (g < nh) {
                float part = 0.f;
                for (int d = lane; d < hd; d += 32) part = fmaf(qs[g * hd + d], to_f32(kr[d]), part);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
                const float mn = fmaxf(m[g], part);
                const float alpha = exp2f(m[g] - mn);
                const float p = exp2f(part - mn);
                l[g] = fmaf(l[g], alpha, p);
                m[g] = mn;
                for (int d = lane; d < hd; d += 32)
                    acc[g * hd + d] = fmaf(p, to_f32(vr[d]), acc[g * hd + d] * alpha);
            }
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < kGenMaxHeads; ++g)
            if (g < nh) {
                ms[warp * hpc + g] = m[g];
                ls[warp * hpc + g] = l[g];
            }
    }
    __syncthreads();

    for (int t = threadIdx.x; t < nh * hd; t += blockDim.x) {
        const int g = t / hd, d = t - g * hd;
        float M = -INFINITY;
        for (int w = 0; w < kGenW; ++w) M = fmaxf(M, ms[w * hpc + g]);
        float num = 0.f, den = 0.f;
        for (int w = 0; w < kGenW; ++w) {
            const float mw = ms[w * hpc + g];
            if (mw != -INFINITY) {
                const float wt = exp2f(mw - M);
                num = fmaf(wt, accs[(w * hpc + g) * hd + d], num);
                den = fmaf(wt, ls[w * hpc + g], den);
            }
        }
        const int h = h0 + g;
        if (u.item < 0) {
            a.out[static_cast<size_t>(rd.q_row0 + u.qi) * (a.n_heads * hd) +
                  static_cast<size_t>(h) * hd + d] = num * ks / den;
        } else {
            const size_t ph = static_cast<size_t>(a.merges[u.item].part0 + u.split) * a.n_heads + h;
            a.pacc[ph * hd + d] = num * ks;
            if (d == 0) {
                a.pm[ph] = M;
                a.pl[ph] = den;
            }
        }
    }
}

// ------------------------------------------------------------------ merge ----

// One warp per (query, head): out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s,
// splits taken in ascending order.
__global__ void merge_splits_kernel(MergeArgs a) {
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= a.n_items * a.n_heads) return;
    const int it = gw / a.n_heads, h = gw - it * a.n_heads;
    const MergeDesc md = a.items[it];
    const RowDesc rd = a.rows[md.row];
    float M = -INFINITY;
    for (int s = 0; s < md.n_split; ++s)
        M = fmaxf(M, a.pm[static_cast<size_t>(md.part0 + s) * a.n_heads + h]);
    float den = 0.f;
    for (int s = 0; s < md.n_split; ++s) {
        const size_t ph = static_cast<size_t>(md.part0 + s) * a.n_heads + h;
        den = fmaf(exp2f(a.pm[ph] - M), a.pl[ph], den);
    }
    float *o = a.out + static_cast<size_t>(rd.q_row0 + md.qi) * (a.n_heads * a.hd) +
               static_cast<size_t>(h) * a.hd;
    const bool vec = (a.hd & 3) == 0 && ((reinterpret_cast<uintptr_t>(a.pacc) |
                                           reinterpret_cast<uintptr_t>(o)) & 15) == 0;
    if (vec) {
        // lane owns 4 consecutive dims: the splits' float4 loads are
        // independent and in flight together (same sums, same order)
        for (int d4 = lane; 4 * d4 < a.hd; d4 += 32) {
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int s = 0; s < md.n_split; ++s) {
                const size_t ph = static_cast<size_t>(md.part0 + s) * a.n_heads + h;
                num = fma4(exp2f(a.pm[ph] - M), ldg4(a.pacc + ph * a.hd + 4 * d4), num);
            }
            reinterpret_cast<float4 *>(o)[d4] = make_float4(num.x / den, num.y / den, num.z / den,
                                                            num.w / den);
        }
        return;
    }
    for (int d = lane; d < a.hd; d += 32) {
        float num = 0.f;
        for (int s = 0; s < md.n_split; ++s) {
            const size_t ph = static_cast<size_t>(md.part0 + s) * a.n_heads + h;
            num = fmaf(exp2f(a.pm[ph] - M), a.pacc[ph * a.hd + d], num);
        }
        o[d] = num / den;
    }
}

// -------------------------------------------------------------- dispatch ----

#ifndef PKV_FAST_STAGES
#define PKV_FAST_STAGES 2
#endif
constexpr int kFastStages = PKV_FAST_STAGES;

template <int G, class Rows>
cudaError_t launch_fast(const AttnArgs &a, const Rows &r, cudaStream_t s) {
    constexpr size_t smem = fast_smem_bytes<G, kFastStages, typename Rows::Elem>();
    static PerDeviceOnce configured;  // the attribute is per function and device
    const cudaError_t ce = configured.run([&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(decode_fast_kernel<G, kFastStages, Rows>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        return cudaSuccess;
    });
    if (ce != cudaSuccess) return ce;
    const long long grid = static_cast<long long>(a.n_units) * a.n_kv;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    decode_fast_kernel<G, kFastStages, Rows><<<static_cast<unsigned>(grid), 128, smem, s>>>(a, r);
    return cudaGetLastError();
}

template <class Rows>
cudaError_t launch_generic(const AttnArgs &a, const Rows &r, cudaStream_t s) {
    const int hpc = a.group < kGenMaxHeads ? a.group : kGenMaxHeads;
    const size_t smem = generic_smem_floats(hpc, a.hd) * sizeof(float);
    static PerDeviceOnce configured;  // the attribute is per function and device
    const cudaError_t ce = configured.run([&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(decode_generic_kernel<Rows>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(generic_smem_floats(kGenMaxHeads, kMaxHeadDim) * sizeof(float)));
        if (e != cudaSuccess) return e;
        return cudaSuccess;
    });
    if (ce != cudaSuccess) return ce;
    const int n_chunks = (a.group + hpc - 1) / hpc;
    const long long grid = static_cast<long long>(a.n_units) * a.n_kv * n_chunks;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    decode_generic_kernel<Rows><<<static_cast<unsigned>(grid), 128, smem, s>>>(a, r, hpc);
    return cudaGetLastError();
}

template <class Rows>
cudaError_t launch_decode(const AttnArgs &a, const Rows &r, cudaStream_t s) {
    if (a.hd == 128) {
        if (a.group == 4) return launch_fast<4>(a, r, s);
        if (a.group == 2) return launch_fast<2>(a, r, s);
        if (a.group == 1) return launch_fast<1>(a, r, s);
    }
    return launch_generic(a, r, s);
}

}  // namespace

cudaError_t launch_pt_apply(int32_t *pt_dev, int32_t max_blocks, const PtRun *runs, int32_t n_runs,
                            const int32_t *vals, cudaStream_t s) {
    if (n_runs <= 0) return cudaSuccess;
    pt_apply_kernel<<<n_runs, 128, 0, s>>>(pt_dev, max_blocks, runs, vals);
    return cudaGetLastError();
}

cudaError_t launch_prep(const PrepArgs &p, const PagedAddr &addr, cudaStream_t s) {
    const long long app_blocks = ((p.rope_base > 0.0 ? 3LL : 2LL) * p.n_app + 7) / 8;
    const long long grid = p.n_runs + app_blocks;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prep_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(p, addr);
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void *kp, void *vp, const CopyDesc *items, int32_t n_items,
                               int64_t block_floats, int32_t n_blocks, int32_t *err,
                               cudaStream_t s) {
    float *k = static_cast<float *>(kp), *v = static_cast<float *>(vp);
    if (n_items <= 0) return cudaSuccess;
    const long long per = (block_floats + 3) / 4;
    unsigned bx = static_cast<unsigned>((per + 255) / 256);
    if (bx > 64) bx = 64;
    if (bx == 0) bx = 1;
    dim3 grid(bx, static_cast<unsigned>(n_items));
    copy_blocks_kernel<<<grid, 256, 0, s>>>(k, v, items, block_floats, n_blocks, err);
    return cudaGetLastError();
}

#ifndef PKV_NARROW_MMA
#define PKV_NARROW_MMA 1
#endif

cudaError_t launch_decode_paged(const AttnArgs &a, const PagedAddr &addr, cudaStream_t s) {
    // bf16 / fp8 pools: the tensor-core decode kernel where it has the shape
    // (the only narrow-pool kernel that takes a fused append)
    if (PKV_NARROW_MMA && decode_mma_shape(a.hd, a.group, addr.bf16 != 0, addr.fp8 != 0))
        return launch_decode_mma_paged(a, addr, s);
    if ((addr.bf16 || addr.fp8) && a.K_new != nullptr) return cudaErrorInvalidValue;
    if (addr.fp8) return launch_decode(a, PagedRows<fp8>{addr}, s);
    if (addr.bf16) return launch_decode(a, PagedRows<bf16>{addr}, s);
    return launch_decode(a, PagedRows<float>{addr}, s);
}

cudaError_t launch_decode_contig(const AttnArgs &a, const ContigAddr &addr, cudaStream_t s) {
    return launch_decode(a, ContigRows{addr}, s);
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s) {
    if (a.n_items <= 0) return cudaSuccess;
    const long long warps = static_cast<long long>(a.n_items) * a.n_heads;
    const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
    merge_splits_kernel<<<blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
