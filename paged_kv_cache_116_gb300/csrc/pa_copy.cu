// pa_copy.cu -- the byte-moving kernels of the path: slot translation, the
// slot-mapped K/V row write (plain, or quantizing into an FP8 cache), and the
// copy-on-write block copy.
//
// All three are HBM-bound moves.  Rows and blocks are moved as 16-byte
// vectors (rows are required to be multiples of 16 bytes), one warp per row
// or a whole CTA per block pair, so every warp instruction touches whole
// 32-byte sectors.
#include <cuda_fp8.h>

#include <algorithm>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Launch as a programmatic dependent of the previous kernel on the stream:
// its launch overlaps that kernel's tail; the kernel waits for it
// (griddepcontrol.wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// slot = block_tables[seq][pos / block_size] * block_size + pos % block_size;
// a negative position gives -1 ("分页 KV Cache", slot_mapping_for).
__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int32_t max_blocks,
                                    const int32_t* __restrict__ seq_idx, const int64_t* __restrict__ positions,
                                    int64_t n, int32_t block_size, int64_t* __restrict__ slot_out) {
    pdl_wait_primary();  // launched as a programmatic dependent: inputs may come from the kernel before
    pdl_launch_dependents();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pos = positions[i];
        if (pos < 0) {
            slot_out[i] = -1;
            continue;
        }
        const int64_t logical = pos / block_size;
        const int32_t phys = block_tables[(int64_t)seq_idx[i] * max_blocks + logical];
        slot_out[i] = (int64_t)phys * block_size + (pos - logical * block_size);
    }
}

// One warp per (token, K|V): the token's row of row_vecs 16-byte vectors goes
// to row slot_mapping[token] of the cache ("分页 KV Cache", PagedKVCache.write).
constexpr int kWriteWarps = 8;

__global__ void __launch_bounds__(kWriteWarps * 32)
    write_kv_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
                    int64_t n, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int64_t row_vecs) {
    pdl_wait_primary();  // the slots (or the pool) may come from the kernel before
    // a dependent kernel (the decode reading these rows) may be scheduled
    // now; it waits for this grid to finish before it reads anything
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x * (int64_t)(kWriteWarps / 2) + (warp >> 1);
    if (item >= n) return;
    const int64_t slot = slots[item];
    if (slot < 0) return;
    const uint4* src = (warp & 1) ? v : k;
    uint4* dst = (warp & 1) ? v_cache : k_cache;
    src += item * row_vecs;
    dst += slot * row_vecs;
    for (int64_t e = lane; e < row_vecs; e += 32) dst[e] = ld_nc_v4(src + e);
}

// One warp per (sequence, K|V): the new token's row goes to the slot of
// position L-1, translated through the sequence's block table.
__global__ void __launch_bounds__(kWriteWarps * 32)
    append_kv_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     const int32_t* __restrict__ block_tables, int32_t max_blocks,
                     const int32_t* __restrict__ context_lens, int32_t num_seqs, int32_t block_size,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int64_t row_vecs) {
    pdl_wait_primary();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t s = blockIdx.x * (int64_t)(kWriteWarps / 2) + (warp >> 1);
    if (s >= num_seqs) return;
    const int32_t L = context_lens[s];
    if (L <= 0) return;
    const int64_t pos = L - 1, logical = pos / block_size;
    const int64_t slot = (int64_t)block_tables[s * max_blocks + logical] * block_size + (pos - logical * block_size);
    const uint4* src = ((warp & 1) ? v_new : k_new) + s * row_vecs;
    uint4* dst = ((warp & 1) ? v_cache : k_cache) + slot * row_vecs;
    for (int64_t e = lane; e < row_vecs; e += 32) dst[e] = ld_nc_v4(src + e);
}

// Quantizing write.  scale = max|x| / 448 (1 for an all-zero row), code =
// E4M3(x / scale), nearest with ties to even, held at +-448; the division
// and maximum in fp32 (IEEE).  A row's codes go to its slot of the code pool,
// its scale to [slot / block_size][head][slot % block_size].  Rows are
// (token or sequence, KV head, K|V), numbered item = row * 2 + is_v with
// row = t * hkv + h.
constexpr int kQuantWarps = 8;
constexpr int kQuantMaxCtas = 4096;

// Where row `item` goes: the element source, the code destination and the
// scale slot; false for a skipped token (negative slot, or length 0).
struct QuantDst {
    int64_t src_row;
    uint8_t* codes;
    float* scale;
};
struct SlotRows {  // pa_write_kv_fp8: slots given per token
    const int64_t* slots;
    __device__ bool slot_of(int64_t t, int32_t bs, int64_t& blk, int64_t& off) const {
        const int64_t slot = slots[t];
        if (slot < 0) return false;
        blk = slot / bs;
        off = slot - blk * bs;
        return true;
    }
};
struct AppendRows {  // the generation step: position context_lens[s] - 1 of sequence s
    const int32_t* block_tables;
    int32_t max_blocks;
    const int32_t* context_lens;
    __device__ bool slot_of(int64_t s, int32_t bs, int64_t& blk, int64_t& off) const {
        const int32_t L = context_lens[s];
        if (L <= 0) return false;
        const int64_t pos = L - 1, logical = pos / bs;
        off = pos - logical * bs;
        blk = block_tables[s * max_blocks + logical];
        return true;
    }
};
template <typename Rows>
__device__ __forceinline__ bool quant_dst(const Rows& rows, int64_t item, int32_t hkv, int32_t hd, int32_t bs,
                                          uint8_t* k_codes, uint8_t* v_codes, float* k_scales, float* v_scales,
                                          QuantDst& d) {
    const int is_v = (int)(item & 1);
    const int64_t row = item >> 1, t = row / hkv;
    const int32_t h = (int32_t)(row - t * hkv);
    int64_t blk, off;
    if (!rows.slot_of(t, bs, blk, off)) return false;
    d.src_row = row;
    d.codes = (is_v ? v_codes : k_codes) + ((blk * bs + off) * hkv + h) * hd;
    d.scale = (is_v ? v_scales : k_scales) + (blk * hkv + h) * bs + off;
    return true;
}

// Main form, head_dim = 8 * EPL: eight lanes per row, four rows per warp at a
// time; each lane loads its EPL consecutive elements with vector loads and
// stores its EPL codes with vector stores.
template <int BYTES>
__device__ __forceinline__ void copy_vec(void* dst, const void* src) {
    static_assert(BYTES % 4 == 0, "whole words");
    if constexpr (BYTES % 16 == 0) {
#pragma unroll
        for (int i = 0; i < BYTES / 16; ++i)
            reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
    } else if constexpr (BYTES % 8 == 0) {
#pragma unroll
        for (int i = 0; i < BYTES / 8; ++i)
            reinterpret_cast<uint2*>(dst)[i] = reinterpret_cast<const uint2*>(src)[i];
    } else {
#pragma unroll
        for (int i = 0; i < BYTES / 4; ++i)
            reinterpret_cast<uint32_t*>(dst)[i] = reinterpret_cast<const uint32_t*>(src)[i];
    }
}

template <typename T, int EPL, typename Rows>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_rows8_kernel(const T* __restrict__ k, const T* __restrict__ v, Rows rows, int64_t n_items, int32_t hkv,
                       int32_t bs, uint8_t* __restrict__ k_codes, uint8_t* __restrict__ v_codes,
                       float* __restrict__ k_scales, float* __restrict__ v_scales) {
    pdl_wait_primary();
    pdl_launch_dependents();
    constexpr int HD = 8 * EPL;
    const int lane = threadIdx.x & 31, sub = lane >> 3, l8 = lane & 7;
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t q = blockIdx.x * (int64_t)kQuantWarps + (threadIdx.x >> 5); q * 4 < n_items; q += nwarps) {
        const int64_t item = q * 4 + sub;
        QuantDst d;
        const bool live = item < n_items && quant_dst(rows, item, hkv, HD, bs, k_codes, v_codes, k_scales, v_scales, d);
        float x[EPL];
        float amax = 0.f;
        if (live) {
            T e[EPL];
            copy_vec<EPL * (int)sizeof(T)>(e, ((item & 1) ? v : k) + d.src_row * HD + l8 * EPL);
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                x[i] = Elt<T>::to_f(e[i]);
                amax = fmaxf(amax, fabsf(x[i]));
            }
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (!live) continue;
        const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        uint32_t c[EPL / 4];
#pragma unroll
        for (int i = 0; i < EPL / 4; ++i) {
            c[i] = 0u;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                c[i] |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[4 * i + t], s), __NV_SATFINITE, __NV_E4M3)
                        << (8 * t);
        }
        copy_vec<EPL>(d.codes + l8 * EPL, c);
        if (l8 == 0) *d.scale = s;
    }
}

// Any head_dim <= 256: one warp per row, element by element.
template <typename T, typename Rows>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_rows_kernel(const T* __restrict__ k, const T* __restrict__ v, Rows rows, int64_t n_items, int32_t hkv,
                      int32_t hd, int32_t bs, uint8_t* __restrict__ k_codes, uint8_t* __restrict__ v_codes,
                      float* __restrict__ k_scales, float* __restrict__ v_scales) {
    pdl_wait_primary();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t item = blockIdx.x * (int64_t)kQuantWarps + (threadIdx.x >> 5); item < n_items; item += nwarps) {
        QuantDst d;
        if (!quant_dst(rows, item, hkv, hd, bs, k_codes, v_codes, k_scales, v_scales, d)) continue;
        const T* src = ((item & 1) ? v : k) + d.src_row * hd;
        float x[8], amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            x[j] = e < hd ? Elt<T>::to_f(src[e]) : 0.f;
            amax = fmaxf(amax, fabsf(x[j]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane + 32 * j;
            if (e < hd) d.codes[e] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[j], s), __NV_SATFINITE, __NV_E4M3);
        }
        if (lane == 0) *d.scale = s;
    }
}

template <typename T, typename Rows>
cudaError_t launch_quant(const void* k, const void* v, const Rows& rows, int64_t n_items, int32_t hkv, int32_t hd,
                         int32_t bs, uint8_t* k_codes, uint8_t* v_codes, float* k_scales, float* v_scales,
                         cudaStream_t stream) {
    if (n_items == 0) return cudaSuccess;
    const T* kt = static_cast<const T*>(k);
    const T* vt = static_cast<const T*>(v);
    const int64_t per_cta = kQuantWarps * ((hd % 8 == 0 && hd <= 256) ? 4 : 1);
    const unsigned grid = (unsigned)std::min<int64_t>((n_items + per_cta - 1) / per_cta, kQuantMaxCtas);
    const dim3 block(kQuantWarps * 32);
    switch (hd % 8 == 0 ? hd / 8 : 0) {
        case 4: return launch_pdl(quant_rows8_kernel<T, 4, Rows>, grid, block, stream, kt, vt, rows, n_items, hkv, bs, k_codes, v_codes, k_scales, v_scales);
        case 8: return launch_pdl(quant_rows8_kernel<T, 8, Rows>, grid, block, stream, kt, vt, rows, n_items, hkv, bs, k_codes, v_codes, k_scales, v_scales);
        case 16: return launch_pdl(quant_rows8_kernel<T, 16, Rows>, grid, block, stream, kt, vt, rows, n_items, hkv, bs, k_codes, v_codes, k_scales, v_scales);
        case 32: return launch_pdl(quant_rows8_kernel<T, 32, Rows>, grid, block, stream, kt, vt, rows, n_items, hkv, bs, k_codes, v_codes, k_scales, v_scales);
        default: return launch_pdl(quant_rows_kernel<T, Rows>, grid, block, stream, kt, vt, rows, n_items, hkv, hd, bs, k_codes, v_codes, k_scales, v_scales);
    }
    return cudaGetLastError();
}

template <typename Rows>
cudaError_t launch_quant_dtype(int dtype, const void* k, const void* v, const Rows& rows, int64_t n_items,
                               int32_t hkv, int32_t hd, int32_t bs, uint8_t* k_codes, uint8_t* v_codes,
                               float* k_scales, float* v_scales, cudaStream_t stream) {
    switch (dtype) {
        case 0: return launch_quant<float>(k, v, rows, n_items, hkv, hd, bs, k_codes, v_codes, k_scales, v_scales, stream);
        case 1: return launch_quant<__nv_bfloat16>(k, v, rows, n_items, hkv, hd, bs, k_codes, v_codes, k_scales, v_scales, stream);
        default: return launch_quant<__half>(k, v, rows, n_items, hkv, hd, bs, k_codes, v_codes, k_scales, v_scales, stream);
    }
}

// One CTA per (pair, layer); its threads stride over the K and V blocks.
struct CopyPtrs {
    uint4* k[PA_MAX_LAYERS_INTERNAL];
    uint4* v[PA_MAX_LAYERS_INTERNAL];
};

__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const CopyPtrs ptrs, const int64_t* __restrict__ pairs, int64_t block_vecs) {
    pdl_wait_primary();  // the pool may still be read or written by the kernel before
    pdl_launch_dependents();
    const int64_t pair = blockIdx.x;
    const int layer = blockIdx.y;
    const int64_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    const uint4* ks = ptrs.k[layer] + src * block_vecs;
    const uint4* vs = ptrs.v[layer] + src * block_vecs;
    uint4* kd = ptrs.k[layer] + dst * block_vecs;
    uint4* vd = ptrs.v[layer] + dst * block_vecs;
    for (int64_t e = threadIdx.x; e < block_vecs; e += blockDim.x) {
        const uint4 a = ld_nc_v4(ks + e);
        const uint4 b = ld_nc_v4(vs + e);
        kd[e] = a;
        vd[e] = b;
    }
}

// Swap: one CTA per (pair, layer) copies a block between two different
// pools; either side may be pinned host memory reached over NVLink-C2C,
// where a read takes microseconds, so each thread keeps kSwapUnroll K and
// V vectors in flight before it stores them.
struct SwapPtrs {
    const uint4* src_k[PA_MAX_LAYERS_INTERNAL];
    const uint4* src_v[PA_MAX_LAYERS_INTERNAL];
    uint4* dst_k[PA_MAX_LAYERS_INTERNAL];
    uint4* dst_v[PA_MAX_LAYERS_INTERNAL];
};

constexpr int kSwapUnroll = 4;

__global__ void __launch_bounds__(256)
    swap_blocks_kernel(const SwapPtrs ptrs, const int64_t* __restrict__ pairs, int64_t block_vecs) {
    const int64_t pair = blockIdx.x;
    const int layer = blockIdx.y;
    const int64_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    const uint4* ks = ptrs.src_k[layer] + src * block_vecs;
    const uint4* vs = ptrs.src_v[layer] + src * block_vecs;
    uint4* kd = ptrs.dst_k[layer] + dst * block_vecs;
    uint4* vd = ptrs.dst_v[layer] + dst * block_vecs;
    for (int64_t base = threadIdx.x; base < block_vecs; base += kSwapUnroll * blockDim.x) {
        uint4 a[kSwapUnroll], b[kSwapUnroll];
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const int64_t e = base + (int64_t)u * blockDim.x;
            if (e < block_vecs) {
                a[u] = ks[e];
                b[u] = vs[e];
            }
        }
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const int64_t e = base + (int64_t)u * blockDim.x;
            if (e < block_vecs) {
                kd[e] = a[u];
                vd[e] = b[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k, void* const* dst_v,
                               int32_t num_layers, const int64_t* block_pairs, int32_t num_pairs, int64_t block_bytes,
                               cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    SwapPtrs ptrs;
    for (int l = 0; l < num_layers; ++l) {
        ptrs.src_k[l] = static_cast<const uint4*>(src_k[l]);
        ptrs.src_v[l] = static_cast<const uint4*>(src_v[l]);
        ptrs.dst_k[l] = static_cast<uint4*>(dst_k[l]);
        ptrs.dst_v[l] = static_cast<uint4*>(dst_v[l]);
    }
    dim3 grid((unsigned)num_pairs, (unsigned)num_layers);
    swap_blocks_kernel<<<grid, 256, 0, stream>>>(ptrs, block_pairs, block_bytes / 16);
    return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_idx,
                                const int64_t* positions, int64_t n, int32_t block_size, int64_t* slot_out,
                                cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    return launch_pdl(slot_mapping_kernel, dim3((unsigned)(blocks < 65535 ? blocks : 65535)), dim3(threads), stream,
                      block_tables, max_blocks, seq_idx, positions, n, block_size, slot_out);
}

cudaError_t launch_write_kv(const void* k, const void* v, const int64_t* slot_mapping, int64_t n, void* k_cache,
                            void* v_cache, int64_t row_bytes, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int64_t per_cta = kWriteWarps / 2;
    const int64_t blocks = (n + per_cta - 1) / per_cta;
    return launch_pdl(write_kv_kernel, dim3((unsigned)blocks), dim3(kWriteWarps * 32), stream,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, n,
                      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), row_bytes / 16);
}

cudaError_t launch_append_kv(const void* k_new, const void* v_new, const int32_t* block_tables, int32_t max_blocks,
                             const int32_t* context_lens, int32_t num_seqs, int32_t block_size, void* k_cache,
                             void* v_cache, int64_t row_bytes, cudaStream_t stream) {
    if (num_seqs == 0) return cudaSuccess;
    const int64_t per_cta = kWriteWarps / 2;
    return launch_pdl(append_kv_kernel, dim3((unsigned)((num_seqs + per_cta - 1) / per_cta)), dim3(kWriteWarps * 32),
                      stream, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables,
                      max_blocks, context_lens, num_seqs, block_size, static_cast<uint4*>(k_cache),
                      static_cast<uint4*>(v_cache), row_bytes / 16);
}

cudaError_t launch_write_kv_fp8(const void* k, const void* v, int dtype, const int64_t* slot_mapping, int64_t n,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, uint8_t* k_codes,
                                uint8_t* v_codes, float* k_scales, float* v_scales, cudaStream_t stream) {
    return launch_quant_dtype(dtype, k, v, SlotRows{slot_mapping}, n * num_kv_heads * 2, num_kv_heads, head_dim,
                              block_size, k_codes, v_codes, k_scales, v_scales, stream);
}

cudaError_t launch_append_kv_fp8(const void* k_new, const void* v_new, int dtype, const int32_t* block_tables,
                                 int32_t max_blocks, const int32_t* context_lens, int32_t num_seqs,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size, uint8_t* k_codes,
                                 uint8_t* v_codes, float* k_scales, float* v_scales, cudaStream_t stream) {
    return launch_quant_dtype(dtype, k_new, v_new, AppendRows{block_tables, max_blocks, context_lens},
                              (int64_t)num_seqs * num_kv_heads * 2, num_kv_heads, head_dim, block_size, k_codes,
                              v_codes, k_scales, v_scales, stream);
}

cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                               const int64_t* block_pairs, int32_t num_pairs, int64_t block_bytes,
                               cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    CopyPtrs ptrs;
    for (int l = 0; l < num_layers; ++l) {
        ptrs.k[l] = static_cast<uint4*>(k_caches[l]);
        ptrs.v[l] = static_cast<uint4*>(v_caches[l]);
    }
    dim3 grid((unsigned)num_pairs, (unsigned)num_layers);
    return launch_pdl(copy_blocks_kernel, grid, dim3(256), stream, ptrs, block_pairs, block_bytes / 16);
}

}  // namespace pa
