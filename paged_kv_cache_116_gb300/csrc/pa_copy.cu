// pa_copy.cu -- the byte-moving kernels of the path: slot translation, the
// slot-mapped K/V row write (plain, or quantizing into an FP8 cache), and the
// copy-on-write block copy.
//
// All three are HBM-bound moves.  Rows and blocks are moved as 16-byte
// vectors (rows are required to be multiples of 16 bytes), one warp per row
// or a whole CTA per block pair, so every warp instruction touches whole
// 32-byte sectors.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

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

// Quantizing write: one warp per (token, KV head, K|V) row of head_dim <=
// 256 elements.  scale = max|x| / 448 (1 for an all-zero row), code =
// E4M3(x / scale), nearest with ties to even, held at +-448; the division
// and maximum in fp32 (IEEE).  The codes go to the row's slot of the code
// pool, the scale to [slot / block_size][head][slot % block_size].
constexpr int kQuantWarps = 8;

// One warp quantizes one row of hd <= 256 elements (src in T) into codes at
// dst and its scale at *scale.
template <typename T>
__device__ __forceinline__ void quantize_row(const T* __restrict__ src, int32_t hd, uint8_t* __restrict__ dst,
                                             float* __restrict__ scale, int lane) {
    float x[8], amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int d = lane + 32 * j;
        x[j] = d < hd ? Elt<T>::to_f(src[d]) : 0.f;
        amax = fmaxf(amax, fabsf(x[j]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int d = lane + 32 * j;
        if (d < hd) dst[d] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[j], s), __NV_SATFINITE, __NV_E4M3);
    }
    if (lane == 0) *scale = s;
}

// Warp item -> (token or sequence, KV head, K|V): item = (row * 2 + is_v), row = t * hkv + h.
template <typename T>
__global__ void __launch_bounds__(kQuantWarps * 32)
    write_kv_fp8_kernel(const T* __restrict__ k, const T* __restrict__ v, const int64_t* __restrict__ slots,
                        int64_t n, int32_t hkv, int32_t hd, int32_t bs, uint8_t* __restrict__ k_codes,
                        uint8_t* __restrict__ v_codes, float* __restrict__ k_scales, float* __restrict__ v_scales) {
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x * (int64_t)kQuantWarps + warp;
    if (item >= n * hkv * 2) return;
    const int is_v = (int)(item & 1);
    const int64_t row = item >> 1, token = row / hkv;
    const int32_t h = (int32_t)(row - token * hkv);
    const int64_t slot = slots[token];
    if (slot < 0) return;
    const int64_t blk = slot / bs;
    quantize_row((is_v ? v : k) + row * hd, hd, (is_v ? v_codes : k_codes) + (slot * hkv + h) * hd,
                 (is_v ? v_scales : k_scales) + (blk * hkv + h) * bs + (slot - blk * bs), lane);
}

// The generation step's quantizing write: sequence s's new rows k_new[s],
// v_new[s] go to the slot of position context_lens[s] - 1 (length-0
// sequences are skipped).
template <typename T>
__global__ void __launch_bounds__(kQuantWarps * 32)
    append_kv_fp8_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new,
                         const int32_t* __restrict__ block_tables, int32_t max_blocks,
                         const int32_t* __restrict__ context_lens, int32_t num_seqs, int32_t hkv, int32_t hd,
                         int32_t bs, uint8_t* __restrict__ k_codes, uint8_t* __restrict__ v_codes,
                         float* __restrict__ k_scales, float* __restrict__ v_scales) {
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x * (int64_t)kQuantWarps + warp;
    if (item >= (int64_t)num_seqs * hkv * 2) return;
    const int is_v = (int)(item & 1);
    const int64_t row = item >> 1, s = row / hkv;
    const int32_t h = (int32_t)(row - s * hkv);
    const int32_t L = context_lens[s];
    if (L <= 0) return;
    const int64_t pos = L - 1, logical = pos / bs, off = pos - logical * bs;
    const int64_t blk = block_tables[s * max_blocks + logical], slot = blk * bs + off;
    quantize_row((is_v ? v_new : k_new) + row * hd, hd, (is_v ? v_codes : k_codes) + (slot * hkv + h) * hd,
                 (is_v ? v_scales : k_scales) + (blk * hkv + h) * bs + off, lane);
}

// One CTA per (pair, layer); its threads stride over the K and V blocks.
struct CopyPtrs {
    uint4* k[PA_MAX_LAYERS_INTERNAL];
    uint4* v[PA_MAX_LAYERS_INTERNAL];
};

__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const CopyPtrs ptrs, const int64_t* __restrict__ pairs, int64_t block_vecs) {
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
    slot_mapping_kernel<<<(unsigned)(blocks < 65535 ? blocks : 65535), threads, 0, stream>>>(
        block_tables, max_blocks, seq_idx, positions, n, block_size, slot_out);
    return cudaGetLastError();
}

cudaError_t launch_write_kv(const void* k, const void* v, const int64_t* slot_mapping, int64_t n, void* k_cache,
                            void* v_cache, int64_t row_bytes, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int64_t per_cta = kWriteWarps / 2;
    const int64_t blocks = (n + per_cta - 1) / per_cta;
    write_kv_kernel<<<(unsigned)blocks, kWriteWarps * 32, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, n, static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), row_bytes / 16);
    return cudaGetLastError();
}

cudaError_t launch_append_kv(const void* k_new, const void* v_new, const int32_t* block_tables, int32_t max_blocks,
                             const int32_t* context_lens, int32_t num_seqs, int32_t block_size, void* k_cache,
                             void* v_cache, int64_t row_bytes, cudaStream_t stream) {
    if (num_seqs == 0) return cudaSuccess;
    const int64_t per_cta = kWriteWarps / 2;
    append_kv_kernel<<<(unsigned)((num_seqs + per_cta - 1) / per_cta), kWriteWarps * 32, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), block_tables, max_blocks, context_lens,
        num_seqs, block_size, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), row_bytes / 16);
    return cudaGetLastError();
}

cudaError_t launch_write_kv_fp8(const void* k, const void* v, int dtype, const int64_t* slot_mapping, int64_t n,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, uint8_t* k_codes,
                                uint8_t* v_codes, float* k_scales, float* v_scales, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int64_t rows = n * num_kv_heads * 2;
    const unsigned blocks = (unsigned)((rows + kQuantWarps - 1) / kQuantWarps);
#define PA_QW(T)                                                                                               \
    write_kv_fp8_kernel<T><<<blocks, kQuantWarps * 32, 0, stream>>>(                                         \
        static_cast<const T*>(k), static_cast<const T*>(v), slot_mapping, n, num_kv_heads, head_dim, block_size, \
        k_codes, v_codes, k_scales, v_scales)
    switch (dtype) {
        case 0: PA_QW(float); break;
        case 1: PA_QW(__nv_bfloat16); break;
        default: PA_QW(__half); break;
    }
#undef PA_QW
    return cudaGetLastError();
}

cudaError_t launch_append_kv_fp8(const void* k_new, const void* v_new, int dtype, const int32_t* block_tables,
                                 int32_t max_blocks, const int32_t* context_lens, int32_t num_seqs,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size, uint8_t* k_codes,
                                 uint8_t* v_codes, float* k_scales, float* v_scales, cudaStream_t stream) {
    if (num_seqs == 0) return cudaSuccess;
    const int64_t rows = (int64_t)num_seqs * num_kv_heads * 2;
    const unsigned blocks = (unsigned)((rows + kQuantWarps - 1) / kQuantWarps);
#define PA_QA(T)                                                                                              \
    append_kv_fp8_kernel<T><<<blocks, kQuantWarps * 32, 0, stream>>>(                                       \
        static_cast<const T*>(k_new), static_cast<const T*>(v_new), block_tables, max_blocks, context_lens,  \
        num_seqs, num_kv_heads, head_dim, block_size, k_codes, v_codes, k_scales, v_scales)
    switch (dtype) {
        case 0: PA_QA(float); break;
        case 1: PA_QA(__nv_bfloat16); break;
        default: PA_QA(__half); break;
    }
#undef PA_QA
    return cudaGetLastError();
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
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(ptrs, block_pairs, block_bytes / 16);
    return cudaGetLastError();
}

}  // namespace pa
