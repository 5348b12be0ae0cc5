// pa_attn_simt.cu -- CUDA-core paged attention for any element type and any
// head_dim up to 256: one CTA per (query row, query head).
//
// This is the path for fp32 (where the 1e-5 bound rules out 16-bit tensor
// operands) and for shapes the tensor-core kernels do not take.  It follows
// the handbook's paged_attention row by row: the row's request comes from
// cu_seqlens_q, its position from seq_len - num_new + j, and its keys are
// read through the block table in logical order.  Each of the CTA's warps
// keeps an online-softmax state over an interleaved share of the keys
// (lanes split head_dim), and the warps' states are merged by their
// log-sum-exp at the end ("aiqz.cc PagedAttention", §工程实现要点: per-block
// softmax merged online).
//
// With a quantized cache (FP8 E4M3 codes, one fp32 scale per token and KV
// head, scales [num_blocks, num_kv_heads, block_size]) a key or value element
// is its code's value times its row's scale; the row scale multiplies the
// dot product of the codes (keys) and the softmax weight (values).
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxDimsPerLane = 8;  // head_dim <= 256

// Cached element -> float: T itself, or (FP8) the value of an E4M3 code.
template <typename T, bool FP8> struct CacheElt {
    using S = T;
    static __device__ __forceinline__ float to_f(S x) { return Elt<T>::to_f(x); }
};
template <typename T> struct CacheElt<T, true> {
    using S = uint8_t;
    static __device__ __forceinline__ float to_f(S x) {
        return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)x, __NV_E4M3)));
    }
};

template <typename T, bool FP8>
__global__ void __launch_bounds__(kWarps * 32) attn_simt_kernel(AttnArgs a) {
    using C = CacheElt<T, FP8>;
    const int row = blockIdx.x;   // query row
    const int head = blockIdx.y;  // query head
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // request of this row: the last i with cu_seqlens_q[i] <= row
    int req = row;
    int num_new = 1, j = 0;
    if (a.cu_seqlens_q != nullptr) {
        int lo = 0, hi = a.num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_seqlens_q[mid] <= row) lo = mid;
            else hi = mid - 1;
        }
        req = lo;
        const int start = a.cu_seqlens_q[req];
        num_new = a.cu_seqlens_q[req + 1] - start;
        j = row - start;
    }
    const int seq_len = a.seq_lens[req];
    const int pos = seq_len - num_new + j;
    const int visible = a.causal ? pos + 1 : seq_len;

    const int G = a.num_heads / a.num_kv_heads;
    const int kvh = head / G;
    const int hd = a.head_dim;
    const int64_t row_elts = (int64_t)a.num_kv_heads * hd;
    const T* q = static_cast<const T*>(a.q) + ((int64_t)row * a.num_heads + head) * hd;
    const typename C::S* kc = static_cast<const typename C::S*>(a.k_cache) + (int64_t)kvh * hd;
    const typename C::S* vc = static_cast<const typename C::S*>(a.v_cache) + (int64_t)kvh * hd;
    const int32_t* table = a.block_tables + (int64_t)req * a.max_blocks;
    const float scale_log2 = a.scale * 1.4426950408889634f;

    float qv[kMaxDimsPerLane], acc[kMaxDimsPerLane];
#pragma unroll
    for (int k = 0; k < kMaxDimsPerLane; ++k) {
        const int d = lane + 32 * k;
        qv[k] = d < hd ? Elt<T>::to_f(q[d]) : 0.f;
        acc[k] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int t = warp; t < visible; t += kWarps) {
        const int64_t blk = table[t / a.block_size], off_in = t % a.block_size;
        const int64_t slot = blk * a.block_size + off_in;
        float ks = 1.f, vs = 1.f;
        if constexpr (FP8) {
            const int64_t si = (blk * a.num_kv_heads + kvh) * a.block_size + off_in;
            ks = a.k_scales[si];
            vs = a.v_scales[si];
        }
        const typename C::S* kr = kc + slot * row_elts;
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxDimsPerLane; ++k) {
            const int d = lane + 32 * k;
            if (d < hd) dot = fmaf(qv[k], C::to_f(kr[d]), dot);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float x = dot * ks * scale_log2;
        const float m_new = fmaxf(m, x);
        const float corr = exp2f(m - m_new);
        const float p = exp2f(x - m_new);
        l = l * corr + p;
        const float pv = p * vs;
        const typename C::S* vr = vc + slot * row_elts;
#pragma unroll
        for (int k = 0; k < kMaxDimsPerLane; ++k) {
            const int d = lane + 32 * k;
            if (d < hd) acc[k] = fmaf(pv, C::to_f(vr[d]), acc[k] * corr);
        }
        m = m_new;
    }

    // merge the warps' (m, l, acc) by their log-sum-exp
    __shared__ float sm_m[kWarps], sm_l[kWarps];
    __shared__ float sm_acc[kWarps][kMaxDimsPerLane * 32];
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
    }
#pragma unroll
    for (int k = 0; k < kMaxDimsPerLane; ++k) sm_acc[warp][lane + 32 * k] = acc[k];
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w]);
    float wgt[kWarps], L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        wgt[w] = sm_m[w] == -INFINITY ? 0.f : exp2f(sm_m[w] - M);
        L += wgt[w] * sm_l[w];
    }
    T* out = static_cast<T*>(a.out) + ((int64_t)row * a.num_heads + head) * hd;
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) o += wgt[w] * sm_acc[w][d];
        out[d] = Elt<T>::from_f(L > 0.f ? o / L : 0.f);
    }
}

}  // namespace

bool attn_simt_supported(int dtype, int head_dim) {
    return (dtype >= 0 && dtype <= 2) && head_dim >= 1 && head_dim <= 32 * kMaxDimsPerLane;
}

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t stream) {
    if (a.total_q == 0) return cudaSuccess;
    dim3 grid((unsigned)a.total_q, (unsigned)a.num_heads);
    if (a.kv_fp8) {
        switch (a.dtype) {
            case 0: attn_simt_kernel<float, true><<<grid, kWarps * 32, 0, stream>>>(a); break;
            case 1: attn_simt_kernel<__nv_bfloat16, true><<<grid, kWarps * 32, 0, stream>>>(a); break;
            default: attn_simt_kernel<__half, true><<<grid, kWarps * 32, 0, stream>>>(a); break;
        }
        return cudaGetLastError();
    }
    switch (a.dtype) {
        case 0: attn_simt_kernel<float, false><<<grid, kWarps * 32, 0, stream>>>(a); break;
        case 1: attn_simt_kernel<__nv_bfloat16, false><<<grid, kWarps * 32, 0, stream>>>(a); break;
        default: attn_simt_kernel<__half, false><<<grid, kWarps * 32, 0, stream>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace pa
