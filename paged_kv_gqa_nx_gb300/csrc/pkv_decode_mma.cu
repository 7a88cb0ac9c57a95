// pkv_decode_mma.cu -- split-K decode over bf16 and fp8 pools, with the two
// products of every key tile on the tensor cores (warp-level m16n8k16 MMAs,
// f32 accumulation).
//
// The work decomposition is the decode kernel's (pkv_kernels.cu): one CTA of
// 4 warps per (work unit, kv head); warp w takes the unit's key tiles w, w+4,
// ... through a 2-stage cp.async pipeline into its own shared memory, keeps an
// online softmax per query head of the GQA group ("nx_f32_attn_paged.nx
// source", step 3: query head h reads kv head h / group), and the 4 warps'
// states are merged at the end.  With 2-byte or 1-byte K/V elements the
// CUDA-core kernel is bound by the instructions it issues per key (widening,
// dot products, shuffles), not by HBM; here a tile of T keys costs
//
//   S[r][key] = sum_d Qp[r][d] K[key][d]     A = query pieces, B = K rows
//   O[r][d]  += sum_key Pp[r][key] V[key][d] A = probability pieces, B = V rows
//
// 2 * T/8 * 8 MMAs, K and V read from shared memory by ldmatrix.  The 16 MMA
// rows r carry the group's query heads split into 16-bit pieces whose sum is
// the f32 value, so the products keep f32 accuracy although the operands are
// 16-bit:
//   bf16 pools: x = p0 + p1 + p2, three bf16 (exact for normal x); for head
//     h < 4 the rows are h (p0), h + 8 (p1) and h + 4 (p2);
//   fp8 pools: x = p0 + p1, two f16 (22 significant bits); rows h (p0) and
//     h + 8 (p1) for h < 8.  e4m3 values are exact in f16.  Each head's query
//     is scaled by a power of two that puts its largest entry in [2^14, 2^15)
//     and P (at most 2^8, see below) by 2^6, so the f16 pieces keep their
//     range; S and O are scaled back exactly.
// K and V elements are exact in the MMA type.  The S accumulator fragment of
// a tile holds, key for key, the A fragment of the PV product (rows gid and
// gid + 8, keys 2*tig, 2*tig + 1 and +8), so P never leaves registers.
//
// The running max of a head moves only when a tile's score passes it by more
// than 8 (base-2 units), so the accumulators are rescaled on few tiles; the
// exponentials, the sum and the merged partials all use the same max, which
// leaves the result unchanged.
//
// Shared memory rows are stored with their 16-byte chunks XOR-swizzled by
// (key & 7), so that the 8 row addresses of every ldmatrix fall in distinct
// bank groups.  Keys past the end of a unit are zero-filled (their scores are
// masked; a zero V row keeps 0 * V finite).
#include "pkv_elem.h"
#include "pkv_internal.h"
#include "pkv_rows.h"

#include <cuda_fp16.h>
#include <type_traits>

namespace pkv {
namespace {

template <class E>
struct MmaCfg;
template <>
struct MmaCfg<bf16> {
    static constexpr int T = 16;  // keys per tile
};
template <>
struct MmaCfg<fp8> {
    static constexpr int T = 32;
};

constexpr int kMmaW = 4;       // warps per CTA
constexpr float kMaxGrow = 8.f;  // log2 headroom of the lazily updated running max
constexpr float kPScale = 64.f;  // f16 probability pieces: p * 2^6 <= 2^14
constexpr int kMmaStages = 2;  // cp.async stages per warp
constexpr int kHD = 128;

template <class E>
__host__ __device__ constexpr int mma_stage_bytes() {
    return MmaCfg<E>::T * kHD * static_cast<int>(sizeof(E)) * 2;  // K rows, then V rows
}
template <class E>
constexpr size_t mma_smem_bytes() {
    return static_cast<size_t>(kMmaW) * kMmaStages * mma_stage_bytes<E>();
}

// D += A * B, m16n8k16, f32 accumulators; bf16 operands on bf16 pools, f16 on fp8 pools.
template <class E>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<bf16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<fp8>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// four e4m3 values (low byte first) -> two f16x2 (bytes 0, 1 and 2, 3; the
// lower byte in the lower half), exact
__device__ __forceinline__ void e4m3x4_f16x2(uint32_t v, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(v));
}

// cp.async of 16 bytes, zero-filled past the first n (0 or 16) source bytes
__device__ __forceinline__ void cp_async16_n(uint32_t dst, const void *src, uint32_t n) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t pack2(bf16, float lo, float hi) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&t);
}
__device__ __forceinline__ uint32_t pack2(fp8, float lo, float hi) {
    const __half2 t = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&t);
}

// The pieces that this lane's two MMA rows (gid, gid + 8) carry for value x.
//   bf16: x = p0 + p1 + p2 (each difference is exact in f32, and p2 has at
//   most 8 significant bits); lanes gid < 4 carry (p0, p1), lanes gid >= 4
//   carry (p2, 0).
//   f16: x = p0 + p1 + (residual below 2^-22 |x|); every lane carries (p0, p1).
__device__ __forceinline__ void pieces(bf16, float x, bool upper, float &r0, float &r1) {
    const float p0 = __bfloat162float(__float2bfloat16_rn(x));
    const float d1 = x - p0;
    const float p1 = __bfloat162float(__float2bfloat16_rn(d1));
    r0 = upper ? d1 - p1 : p0;
    r1 = upper ? 0.f : p1;
}
__device__ __forceinline__ void pieces(fp8, float x, bool, float &r0, float &r1) {
    const float p0 = __half2float(__float2half_rn(x));
    r0 = p0;
    r1 = x - p0;  // rounded to f16 when packed
}

// 2^x by the hardware approximation (relative error near 2^-22; results
// below 2^-126 flush to zero).  Arguments here are score - running max <= 8.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e, e in [-126, 127]
    return __int_as_float((e + 127) << 23);
}

template <int G, class E>
__global__ void __launch_bounds__(128, 3) decode_mma_kernel(AttnArgs a, PagedRows<E> rows_of) {
    using C = MmaCfg<E>;
    constexpr bool kF8 = std::is_same<E, fp8>::value;
    constexpr int T = C::T;
    constexpr int NT = T / 8;                 // 8-key n-tiles of S
    constexpr int KS = T / 16;                // 16-key k-steps of PV
    constexpr int RB = kHD * static_cast<int>(sizeof(E));  // bytes of one K (V) row
    constexpr int CPR = RB / 16;              // 16-byte chunks per row: 16 (bf16), 8 (fp8)
    constexpr int EPC = 16 / static_cast<int>(sizeof(E));  // elements per chunk
    constexpr int STAGE = mma_stage_bytes<E>();
    constexpr int W = kMmaW, NST = kMmaStages;
    static_assert(G >= 1 && G <= (kF8 ? 8 : 4), "query heads per kv head");
    static_assert(NST * STAGE >= (G * kHD + 2 * G) * 4, "a warp's stage memory holds its (acc, m, l)");
    extern __shared__ __align__(128) unsigned char smraw[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int ui = blockIdx.x / a.n_kv;
    const int kvh = blockIdx.x - ui * a.n_kv;
    const UnitDesc u = a.units[ui];
    const RowDesc rd = a.rows[u.row];
    const UnitRange ur = unit_range(u, rd, a.causal, a.split_keys);
    const int n_tiles = (ur.kend - ur.kbeg + T - 1) / T;
    const int my_n = warp < n_tiles ? (n_tiles - warp + W - 1) / W : 0;
    unsigned char *wbase = smraw + warp * NST * STAGE;
    const uint32_t wbase_s = static_cast<uint32_t>(__cvta_generic_to_shared(wbase));

    // ---- tile loads --------------------------------------------------------
    // lane -> (key offset cj, K or V, chunk cch) of the copy: one key per pass
    // on bf16 pools (lanes 0-15 K, 16-31 V), two on fp8 pools.  Key j, chunk c
    // of a stage sits at byte j * RB + ((c ^ (j & 7)) << 4).  Positions past
    // the unit (and rows whose page lookup failed, which sets the error flag)
    // are zero-filled by the copy itself.
    constexpr int KPP = 32 / (2 * CPR);
    const int cj = lane / (2 * CPR);
    const int cpart = lane % (2 * CPR);
    const bool cv = cpart >= CPR;
    const int cch = cv ? cpart - CPR : cpart;
    const int csw = cch ^ cj;  // j & 7 = ((i * KPP) & 7) | cj in pass i
    const uint32_t cdst = wbase_s + (cv ? T * RB : 0) + cj * RB;
    const size_t rstride = rows_of.row_stride();
    const bool pages16 = rows_of.whole_tiles(16) && (ur.kbeg & 15) == 0;
    const E *const zsrc = static_cast<const E *>(cv ? rows_of.a.v : rows_of.a.k);  // read by no copy
    // fused append: positions from past_len on are this call's new rows; they
    // come from K_new / V_new (f32), rounded as the append rounds them
    const bool fused = a.K_new != nullptr;
    const int new0 = fused ? rd.past_len : 0x7fffffff;
    const float inv_scale = 1.f / rows_of.a.kv_scale;  // power of two: exact
    // New row `key` of the tile (position pos) -> the stage, in the layout the
    // copies use (chunk c of key j at j * RB + ((c ^ (j & 7)) << 4)): lane l <
    // 2 * CPR converts chunk l % CPR of K (l < CPR) or V with the append's
    // rounding (store4's conversions) and stores its 16 bytes.
    auto put_new = [&](uint32_t stage, int key, int pos) {
        if (lane >= 2 * CPR) return;
        const int half = lane / CPR, c = lane - half * CPR;
        const float *src = (half ? a.V_new : a.K_new) +
                           static_cast<size_t>(rd.q_row0 + (pos - new0)) * rstride +
                           static_cast<size_t>(kvh) * kHD + c * EPC;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < EPC / 4; ++i) {
            float4 x = __ldg(reinterpret_cast<const float4 *>(src) + i);
            if constexpr (kF8) {
                x = make_float4(x.x * inv_scale, x.y * inv_scale, x.z * inv_scale, x.w * inv_scale);
                const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x.x, x.y), __NV_SATFINITE, __NV_E4M3);
                const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x.z, x.w), __NV_SATFINITE, __NV_E4M3);
                w[i] = lo | (hi << 16);
            } else {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
                w[2 * i] = *reinterpret_cast<const uint32_t *>(&lo);
                w[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&hi);
            }
        }
        const uint32_t dst = stage + (half ? T * RB : 0) + key * RB + ((c ^ (key & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
    };
    // One tile's copies.  kNew (a tile that holds this call's new rows): a key
    // slot is written once, by a copy (pool rows; zero past the unit) or, for
    // a new row, by put_new; every other tile takes the copies alone, with no
    // per-key test (this kernel is bound by the instructions it issues).
    auto copy_tile = [&](int pos0, int st, int nv, int nall, auto new_rows) {
        constexpr bool kNew = decltype(new_rows)::value;
        const uint32_t dst0 = cdst + st * STAGE;
        auto skip = [&](int j) { return kNew && j >= nv && j < nall; };
        if (pages16) {
            // 16 positions from a multiple of 16 share one page
#pragma unroll
            for (int g = 0; g < T / 16; ++g) {
                const E *kb, *vb;
                const bool okg = 16 * g < nv && rows_of.row(rd.slot, pos0 + 16 * g, kvh, kHD, kb, vb, a.err);
                const E *b = okg ? (cv ? vb : kb) + cj * rstride + cch * EPC : zsrc;
#pragma unroll
                for (int i = 0; i < 16 / KPP; ++i) {
                    const int jj = 16 * g + i * KPP;
                    if (skip(jj + cj)) continue;
                    const bool ok = okg && jj + cj < nv;
                    cp_async16_n(dst0 + jj * RB + ((csw ^ ((i * KPP) & 7)) << 4),
                                 ok ? b + static_cast<size_t>(i * KPP) * rstride : zsrc, ok ? 16u : 0u);
                }
            }
        } else {
#pragma unroll 1
            for (int jj = 0; jj < T; jj += KPP) {
                const int j = jj + cj;
                if (skip(j)) continue;
                const E *kr, *vr;
                const bool ok = j < nv && rows_of.row(rd.slot, pos0 + j, kvh, kHD, kr, vr, a.err);
                cp_async16_n(cdst - cj * RB + st * STAGE + j * RB + ((cch ^ (j & 7)) << 4),
                             ok ? (cv ? vr : kr) + cch * EPC : zsrc, ok ? 16u : 0u);
            }
        }
        if constexpr (kNew) {
            const uint32_t stage = wbase_s + st * STAGE;
            for (int j = max(nv, 0); j < nall; ++j) put_new(stage, j, pos0 + j);
        }
    };
    auto load_tile = [&](int kl, int st) {
        const int pos0 = ur.kbeg + (warp + kl * W) * T;
        const int nall = min(T, ur.kend - pos0);  // keys of the unit in this tile
        if (pos0 + T > new0)
            copy_tile(pos0, st, min(nall, new0 - pos0), nall, std::true_type{});
        else
            copy_tile(pos0, st, nall, nall, std::false_type{});
    };

    // the first tiles are in flight while the queries are prepared
#pragma unroll
    for (int s = 0; s < NST - 1; ++s) {
        if (s < my_n) load_tile(s, s);
        cp_async_commit();
    }

    // fused append: the unit of the row's last query stores the new rows of
    // its split into the pool (nothing in this launch reads them from there;
    // the first tiles' copies are already in flight), and enters each new
    // page into the device page table
    if (fused && u.qi == rd.n_q - 1) {
        for (int pos = max(ur.kbeg, new0) + warp; pos < ur.kend; pos += W) {
            const int t = pos - new0;
            const AppendDesc ad = a.app[rd.q_row0 + t];
            const size_t o = static_cast<size_t>(rd.q_row0 + t) * rstride + static_cast<size_t>(kvh) * kHD;
            const bool set_pt = a.pt_write && kvh == 0 && (pos == 0 || rows_of.block_start(pos));
            rows_of.store_row(rd.slot, ad.blk, pos, kvh, kHD, a.K_new + o, a.V_new + o, set_pt, lane, a.err);
        }
    }

    // this lane's query head; for bf16, lanes gid >= 4 carry the third piece
    const int h = kF8 ? gid : (gid & 3);
    const bool hv = h < G;
    const bool upper = !kF8 && gid >= 4;
    const E tag{};

    // ---- query pieces: the A fragments of the 8 k-steps of 16 dims --------
    // Logical k (2tig, 2tig+1 | 2tig+8, 2tig+9) of k-step s is dims
    // 16s + (2tig, 2tig+1 | 8+2tig, 9+2tig) on bf16 pools, and 16s + 4tig + (0,
    // 1 | 2, 3) on fp8 pools (the order in which ldmatrix hands out the bytes
    // of a row of e4m3 values).
    const float ks = rows_of.scale();
    const float qs = a.scale_log2 * ks;
    const float *qrow = a.Q + static_cast<size_t>(rd.q_row0 + u.qi) * (a.n_heads * kHD) +
                        static_cast<size_t>(kvh * G + (hv ? h : 0)) * kHD;
    float qv[8][4];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        if constexpr (kF8) {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(qrow + 16 * s + 4 * tig));
            qv[s][0] = t.x, qv[s][1] = t.y, qv[s][2] = t.z, qv[s][3] = t.w;
        } else {
            const float2 t0 = __ldg(reinterpret_cast<const float2 *>(qrow + 16 * s + 2 * tig));
            const float2 t1 = __ldg(reinterpret_cast<const float2 *>(qrow + 16 * s + 8 + 2 * tig));
            qv[s][0] = t0.x, qv[s][1] = t0.y, qv[s][2] = t1.x, qv[s][3] = t1.y;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[s][i] = hv ? qv[s][i] * qs : 0.f;
    }
    // f16 pieces: per-head power-of-two scale (scores are scaled back by qinv)
    float qinv = 1.f;
    if constexpr (kF8) {
        float qmax = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
            for (int i = 0; i < 4; ++i) qmax = fmaxf(qmax, fabsf(qv[s][i]));
        qmax = fmaxf(qmax, __shfl_xor_sync(kFull, qmax, 1));
        qmax = fmaxf(qmax, __shfl_xor_sync(kFull, qmax, 2));
        int eq = 0;
        if (qmax > 0.f && qmax <= 3.4e38f) {
            const int e = ((__float_as_int(qmax) >> 23) & 0xff) - 127;
            eq = min(max(14 - e, -126), 126);
        }
        const float qsc = pow2f(eq);
        qinv = pow2f(-eq);
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[s][i] *= qsc;
    }
    uint32_t qa[8][4];
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            float a0, a1, b0, b1;
            pieces(tag, qv[s][2 * p], upper, a0, a1);
            pieces(tag, qv[s][2 * p + 1], upper, b0, b1);
            qa[s][2 * p] = pack2(tag, a0, b0);      // row gid
            qa[s][2 * p + 1] = pack2(tag, a1, b1);  // row gid + 8
        }

    // ldmatrix row addresses (byte offsets in a stage; the chunk is XORed in)
    //   K, bf16: matrix mi = (n-tile mi >> 1, chunk 2s + (mi & 1))
    //   K, fp8:  matrix mi = (n-tile mi, chunk s)
    //   V, both: matrix mi = (keys 16kk + 8 (mi & 1) .., chunk 2c + (mi >> 1))
    const int mi = lane >> 3, mr = lane & 7;
    const int kkey = kF8 ? lane : ((mi >> 1) * 8 + mr);
    const int kc0 = kF8 ? 0 : (mi & 1);
    const int vkey = (mi & 1) * 8 + mr;
    const int vc0 = mi >> 1;

    float m_run = -INFINITY, l_run = 0.f;
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int k = 0; k < my_n; ++k) {
        const int kn = k + NST - 1;
        if (kn < my_n) load_tile(kn, kn % NST);
        cp_async_commit();
        cp_async_wait<NST - 1>();
        __syncwarp();

        const int pos0 = ur.kbeg + (warp + k * W) * T;
        const int n_valid = min(T, ur.kend - pos0);
        const uint32_t Ks = wbase_s + (k % NST) * STAGE;
        const uint32_t Vs = Ks + T * RB;

        // S = Q K^T over the tile
        float c[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) c[n][0] = c[n][1] = c[n][2] = c[n][3] = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            uint32_t r[4];
            if constexpr (kF8) {
                ldsm4(r, Ks + kkey * RB + ((s ^ (kkey & 7)) << 4));
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    uint32_t b0, b1;
                    e4m3x4_f16x2(r[n], b0, b1);
                    mma16816<E>(c[n], qa[s], b0, b1);
                }
            } else {
                ldsm4(r, Ks + kkey * RB + (((2 * s + kc0) ^ (kkey & 7)) << 4));
                mma16816<E>(c[0], qa[s], r[0], r[1]);
                mma16816<E>(c[1], qa[s], r[2], r[3]);
            }
        }

        // scores of this lane's head at keys 8n + 2tig, 8n + 2tig + 1
        float sv[NT][2];
        float tmax = -INFINITY;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float x = c[n][e] + c[n][e + 2];
                if constexpr (kF8) x *= qinv;
                else x += __shfl_xor_sync(kFull, x, 16);
                sv[n][e] = (8 * n + 2 * tig + e < n_valid) ? x : -INFINITY;
                tmax = fmaxf(tmax, sv[n][e]);
            }
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 2));
        // the running max moves only when a score passes it by more than
        // kMaxGrow (probabilities stay <= 2^kMaxGrow), so most tiles skip the
        // rescale of the accumulators
        const float m_new = tmax > m_run + kMaxGrow ? tmax : m_run;
        const float alpha = m_new == m_run ? 1.f : ex2(m_run - m_new);
        float ps = 0.f;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                sv[n][e] = ex2(sv[n][e] - m_new);
                ps += sv[n][e];
            }
        ps += __shfl_xor_sync(kFull, ps, 1);
        ps += __shfl_xor_sync(kFull, ps, 2);
        l_run = fmaf(l_run, alpha, ps);
        m_run = m_new;
        if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
            for (int n = 0; n < 16; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[n][e] *= alpha;
        }

        // O += P V: the probabilities of keys 16kk + (2tig, 2tig+1 | +8, +9)
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            uint32_t pa[4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const float pscale = kF8 ? kPScale : 1.f;
                float a0, a1, b0, b1;
                pieces(tag, sv[2 * kk + half][0] * pscale, upper, a0, a1);
                pieces(tag, sv[2 * kk + half][1] * pscale, upper, b0, b1);
                pa[2 * half] = pack2(tag, a0, b0);
                pa[2 * half + 1] = pack2(tag, a1, b1);
            }
            const uint32_t vrow = Vs + (16 * kk + vkey) * RB;
            const int vsw = (16 * kk + vkey) & 7;
            if constexpr (kF8) {
                // a 16-byte chunk is 16 dims: the even dims make n-tile 2ch,
                // the odd dims n-tile 2ch + 1
#pragma unroll
                for (int cp = 0; cp < 4; ++cp) {
                    uint32_t r[4];
                    ldsm4t(r, vrow + (((2 * cp + vc0) ^ vsw) << 4));
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int ch = 2 * cp + q;
                        uint32_t ev0, od0, ev1, od1;  // even / odd dims, keys 2tig.. and 2tig+8..
                        e4m3x4_f16x2(__byte_perm(r[2 * q], 0u, 0x3120), ev0, od0);
                        e4m3x4_f16x2(__byte_perm(r[2 * q + 1], 0u, 0x3120), ev1, od1);
                        mma16816<E>(o[2 * ch], pa, ev0, ev1);
                        mma16816<E>(o[2 * ch + 1], pa, od0, od1);
                    }
                }
            } else {
#pragma unroll
                for (int cp = 0; cp < 8; ++cp) {
                    uint32_t r[4];
                    ldsm4t(r, vrow + (((2 * cp + vc0) ^ vsw) << 4));
                    mma16816<E>(o[2 * cp], pa, r[0], r[1]);
                    mma16816<E>(o[2 * cp + 1], pa, r[2], r[3]);
                }
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncwarp();

    // publish this warp's (acc, m, l) in its own (now idle) stage memory
    float *R = reinterpret_cast<float *>(wbase);
    const float osc = kF8 ? ks * (1.f / kPScale) : ks;
    const bool writer = hv && (kF8 || gid < 4);
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        float o0 = o[n][0] + o[n][2], o1 = o[n][1] + o[n][3];
        if constexpr (!kF8) {
            o0 += __shfl_xor_sync(kFull, o0, 16);
            o1 += __shfl_xor_sync(kFull, o1, 16);
        }
        if (writer) {
            float *Rh = R + h * kHD;
            if constexpr (kF8) {
                const int d = 16 * (n >> 1) + 4 * tig + (n & 1);
                Rh[d] = o0 * osc;
                Rh[d + 2] = o1 * osc;
            } else {
                Rh[8 * n + 2 * tig] = o0 * osc;
                Rh[8 * n + 2 * tig + 1] = o1 * osc;
            }
        }
    }
    if (writer && tig == 0) {
        R[G * kHD + h] = m_run;
        R[G * kHD + G + h] = l_run;
    }
    __syncthreads();

    const int d = threadIdx.x;  // 128 threads <-> 128 dims
    auto Rw = [&](int w) { return reinterpret_cast<const float *>(smraw + w * NST * STAGE); };
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float mw[W];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            mw[w] = Rw(w)[G * kHD + g];
            M = fmaxf(M, mw[w]);
        }
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            if (mw[w] != -INFINITY) {
                const float wt = exp2f(mw[w] - M);
                num = fmaf(wt, Rw(w)[g * kHD + d], num);
                den = fmaf(wt, Rw(w)[G * kHD + G + g], den);
            }
        }
        const int hq = kvh * G + g;
        if (u.item < 0) {
            a.out[static_cast<size_t>(rd.q_row0 + u.qi) * (a.n_heads * kHD) + static_cast<size_t>(hq) * kHD + d] =
                num / den;
        } else {
            const size_t ph = static_cast<size_t>(a.merges[u.item].part0 + u.split) * a.n_heads + hq;
            a.pacc[ph * kHD + d] = num;
            if (d == 0) {
                a.pm[ph] = M;
                a.pl[ph] = den;
            }
        }
    }
}

template <int G, class E>
cudaError_t launch_mma(const AttnArgs &a, const PagedAddr &addr, cudaStream_t s) {
    constexpr size_t smem = mma_smem_bytes<E>();
    static PerDeviceOnce configured;  // the attribute is per function and device
    const cudaError_t ce = configured.run([&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<G, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        return cudaSuccess;
    });
    if (ce != cudaSuccess) return ce;
    const long long grid = static_cast<long long>(a.n_units) * a.n_kv;
    if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    decode_mma_kernel<G, E><<<static_cast<unsigned>(grid), 128, smem, s>>>(a, PagedRows<E>{addr});
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_mma_paged(const AttnArgs &a, const PagedAddr &addr, cudaStream_t s) {
    if (!decode_mma_shape(a.hd, a.group, addr.bf16 != 0, addr.fp8 != 0)) return cudaErrorInvalidValue;
    if (addr.fp8) {
        switch (a.group) {
            case 1: return launch_mma<1, fp8>(a, addr, s);
            case 2: return launch_mma<2, fp8>(a, addr, s);
            case 4: return launch_mma<4, fp8>(a, addr, s);
            default: return launch_mma<8, fp8>(a, addr, s);
        }
    }
    switch (a.group) {
        case 1: return launch_mma<1, bf16>(a, addr, s);
        case 2: return launch_mma<2, bf16>(a, addr, s);
        default: return launch_mma<4, bf16>(a, addr, s);
    }
}

}  // namespace pkv
