// pkv_rows.h -- device helpers shared by the decode kernels (pkv_kernels.cu,
// pkv_decode_mma.cu): cp.async, the error flag, row addressing in the paged
// pool and in a contiguous history, and the key range of a split-K work unit.
// Every kernel that attends a unit takes its keys from unit_range, so the
// split boundaries -- multiples of S keys from the row's first decode key --
// are the same whichever kernel runs it.
#pragma once

#include "pkv_elem.h"
#include <type_traits>
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void flag_error(int32_t *err, int code) {
    if (err) atomicOr(err, code);
}

// ------------------------------------------------------------ addressing ----

template <class E>
struct PagedRows {
    using Elem = E;
    PagedAddr a;
    // Row of (slot, pos) for kv head `kvh`; false (and the error flag) when the
    // page index or the block id is out of range -- the access is skipped.
    __device__ __forceinline__ bool row(int slot, int pos, int kvh, int hd, const E *&kr,
                                        const E *&vr, int32_t *err) const {
        const int bi = a.bs_shift >= 0 ? (pos >> a.bs_shift) : (pos / a.bs);
        const int off = pos - bi * a.bs;
        if (bi >= a.max_blocks) {
            flag_error(err, 1);
            return false;
        }
        const int blk = __ldg(a.pt + static_cast<size_t>(slot) * a.max_blocks + bi);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.n_blocks)) {
            flag_error(err, 1);
            return false;
        }
        const size_t o = static_cast<size_t>(blk) * a.block_stride + a.layer_off +
                         static_cast<size_t>(off) * a.kv_dim + static_cast<size_t>(kvh) * hd;
        kr = static_cast<const E *>(a.k) + o;
        vr = static_cast<const E *>(a.v) + o;
        return true;
    }
    // Tiles of T positions starting at a multiple of T stay inside one block
    // when the block size is a multiple of T: row pos0 + j is then row pos0
    // plus j * kv_dim.
    __device__ __forceinline__ bool whole_tiles(int T) const { return (a.bs % T) == 0; }
    __device__ __forceinline__ size_t row_stride() const { return static_cast<size_t>(a.kv_dim); }
    // read value = stored element * scale (a power of two; 1 except on fp8 pools)
    __device__ __forceinline__ float scale() const { return a.kv_scale; }
    __device__ __forceinline__ bool block_start(int pos) const {
        return (a.bs_shift >= 0 ? (pos & (a.bs - 1)) : (pos % a.bs)) == 0;
    }
    // Fused append: store head kvh's hd floats of one new row (K and V) at
    // position pos of block blk, one float4 per lane of the calling warp,
    // rounded to the pool element as the append kernel rounds them;
    // with set_pt, also enter blk as the page of pos.  False (and the error
    // flag) on an out-of-range block id or page index.
    __device__ __forceinline__ bool store_row(int slot, int blk, int pos, int kvh, int hd,
                                              const float *ks, const float *vs, bool set_pt,
                                              int lane, int32_t *err) const {
        const int bi = a.bs_shift >= 0 ? (pos >> a.bs_shift) : (pos / a.bs);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.n_blocks) || bi >= a.max_blocks) {
            if (lane == 0) flag_error(err, 1);
            return false;
        }
        const size_t o = static_cast<size_t>(blk) * a.block_stride + a.layer_off +
                         static_cast<size_t>(pos - bi * a.bs) * a.kv_dim + static_cast<size_t>(kvh) * hd;
        for (int i = lane; 4 * i < hd; i += 32) {
            float4 k4 = ldg4(ks + 4 * i), v4 = ldg4(vs + 4 * i);
            if constexpr (std::is_same<E, fp8>::value) {
                // e4m3 of x / scale, as the append kernel stores it (a power of two: exact)
                const float inv = 1.f / a.kv_scale;
                k4 = make_float4(k4.x * inv, k4.y * inv, k4.z * inv, k4.w * inv);
                v4 = make_float4(v4.x * inv, v4.y * inv, v4.z * inv, v4.w * inv);
            }
            store4(static_cast<E *>(a.k) + o + 4 * i, k4);
            store4(static_cast<E *>(a.v) + o + 4 * i, v4);
        }
        if (set_pt && lane == 0) a.pt[static_cast<size_t>(slot) * a.max_blocks + bi] = blk;
        return true;
    }
};

struct ContigRows {
    using Elem = float;
    ContigAddr a;
    __device__ __forceinline__ bool row(int, int pos, int kvh, int hd, const float *&kr,
                                        const float *&vr, int32_t *) const {
        const size_t o = static_cast<size_t>(pos) * a.kv_dim + static_cast<size_t>(kvh) * hd;
        kr = a.k + o;
        vr = a.v + o;
        return true;
    }
    __device__ __forceinline__ bool whole_tiles(int) const { return true; }
    __device__ __forceinline__ size_t row_stride() const { return static_cast<size_t>(a.kv_dim); }
    __device__ __forceinline__ float scale() const { return 1.f; }
    // contiguous histories are caller-owned: there is no fused append
    __device__ __forceinline__ bool block_start(int) const { return false; }
    __device__ __forceinline__ bool store_row(int, int, int, int, int, const float *, const float *,
                                              bool, int, int32_t *) const {
        return false;
    }
};

// The key range of one work unit.
struct UnitRange {
    int kbeg, kend;
};
__device__ __forceinline__ UnitRange unit_range(const UnitDesc &u, const RowDesc &rd, int causal,
                                                int split_keys) {
    const int total_k = rd.past_len + rd.n_q;
    const int q_pos = total_k - rd.n_q + u.qi;  // offset-causal query position
    const int lim = causal ? q_pos + 1 : total_k;
    const int kbeg = rd.k0 + (u.split - rd.s0) * split_keys;
    const int kend = min(kbeg + split_keys, lim);
    return {kbeg, kend};
}

}  // namespace
}  // namespace pkv
