// pa_attn_simt.cu -- CUDA-core paged attention for any element type and any
// head_dim up to 256: one CTA per (query row, KV head, group of up to 8 of
// that KV head's query heads).
//
// This is the path for fp32 (where the 1e-5 bound rules out 16-bit tensor
// operands) and for shapes the tensor-core kernels do not take.  It follows
// the handbook's paged_attention row by row: the row's request comes from
// cu_seqlens_q, its position from seq_len - num_new + j, and its keys are
// read through the block table in logical order.  The query heads that
// share a KV head are worked together (query-group packing: each K/V row is
// read once for the CTA's heads, not once per head).  Lanes split head_dim
// and hold every head's query slice and output accumulator; each of the
// CTA's warps keeps one online-softmax state per head over an interleaved
// share of the keys, and the warps' states are merged by their log-sum-exp
// at the end ("aiqz.cc PagedAttention", §工程实现要点: per-block softmax
// merged online).
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

// DPL: head dims per lane (head_dim <= 32 DPL); GH: query heads per CTA.
template <typename T, bool FP8, int DPL, int GH>
__global__ void __launch_bounds__(kWarps * 32) attn_simt_kernel(AttnArgs a) {
    using C = CacheElt<T, FP8>;
    const int row = blockIdx.x;  // query row
    const int G = a.num_heads / a.num_kv_heads;
    const int hchunks = (G + GH - 1) / GH;
    const int kvh = blockIdx.y / hchunks;
    const int h0 = kvh * G + (blockIdx.y - kvh * hchunks) * GH;  // first query head of the CTA
    const int nh = min(GH, kvh * G + G - h0);                    // heads of the CTA
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

    const int hd = a.head_dim;
    const int64_t row_elts = (int64_t)a.num_kv_heads * hd;
    const T* q = static_cast<const T*>(a.q) + ((int64_t)row * a.num_heads + h0) * hd;
    const typename C::S* kc = static_cast<const typename C::S*>(a.k_cache) + (int64_t)kvh * hd;
    const typename C::S* vc = static_cast<const typename C::S*>(a.v_cache) + (int64_t)kvh * hd;
    const int32_t* table = a.block_tables + (int64_t)req * a.max_blocks;
    const float scale_log2 = a.scale * 1.4426950408889634f;

    float qv[GH][DPL], acc[GH][DPL], m[GH], l[GH];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int k = 0; k < DPL; ++k) {
            const int d = lane + 32 * k;
            qv[h][k] = (h < nh && d < hd) ? Elt<T>::to_f(q[(int64_t)h * hd + d]) : 0.f;
            acc[h][k] = 0.f;
        }
    }
    // U tokens per warp in flight: their table entries load together, then
    // their K/V rows, so a warp waits for two memory round trips per U
    // tokens rather than per token; they are then folded in in order (as
    // many as the registers hold without spilling)
    constexpr int U = DPL <= 2 ? 4 : (DPL * GH <= 16 ? 2 : 1);
    for (int t0 = warp; t0 < visible; t0 += U * kWarps) {
        int64_t slot[U];
        float ks[U], vs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = min(t0 + u * kWarps, visible - 1);  // in range; unused past `visible`
            const int64_t blk = table[t / a.block_size], off_in = t % a.block_size;
            slot[u] = blk * a.block_size + off_in;
            ks[u] = vs[u] = 1.f;
            if constexpr (FP8) {
                const int64_t si = (blk * a.num_kv_heads + kvh) * a.block_size + off_in;
                ks[u] = a.k_scales[si];
                vs[u] = a.v_scales[si];
            }
        }
        float kx[U][DPL], vx[U][DPL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const typename C::S* kr = kc + slot[u] * row_elts;
            const typename C::S* vr = vc + slot[u] * row_elts;
#pragma unroll
            for (int k = 0; k < DPL; ++k) {
                const int d = lane + 32 * k;
                kx[u][k] = d < hd ? C::to_f(kr[d]) : 0.f;
                vx[u][k] = d < hd ? C::to_f(vr[d]) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (t0 + u * kWarps >= visible) break;  // warp-uniform
            float dot[GH];
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                dot[h] = 0.f;
#pragma unroll
                for (int k = 0; k < DPL; ++k) dot[h] = fmaf(qv[h][k], kx[u][k], dot[h]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int h = 0; h < GH; ++h) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], off);
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float x = dot[h] * ks[u] * scale_log2;
                const float m_new = fmaxf(m[h], x);
                const float corr = exp2f(m[h] - m_new);
                const float p = exp2f(x - m_new);
                l[h] = l[h] * corr + p;
                const float pv = p * vs[u];
#pragma unroll
                for (int k = 0; k < DPL; ++k) acc[h][k] = fmaf(pv, vx[u][k], acc[h][k] * corr);
                m[h] = m_new;
            }
        }
    }

    // merge the warps' (m, l, acc) per head by their log-sum-exp
    __shared__ float sm_m[kWarps][GH], sm_l[kWarps][GH];
    __shared__ float sm_acc[kWarps][GH][DPL * 32];
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            sm_m[warp][h] = m[h];
            sm_l[warp][h] = l[h];
        }
    }
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
        for (int k = 0; k < DPL; ++k) sm_acc[warp][h][lane + 32 * k] = acc[h][k];
    __syncthreads();
    for (int e = threadIdx.x; e < nh * hd; e += blockDim.x) {
        const int h = e / hd, d = e - h * hd;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][h]);
        float L = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float wgt = sm_m[w][h] == -INFINITY ? 0.f : exp2f(sm_m[w][h] - M);
            L += wgt * sm_l[w][h];
            o += wgt * sm_acc[w][h][d];
        }
        static_cast<T*>(a.out)[((int64_t)row * a.num_heads + h0 + h) * hd + d] = Elt<T>::from_f(L > 0.f ? o / L : 0.f);
    }
}

template <typename T, bool FP8>
cudaError_t launch_typed(const AttnArgs& a, cudaStream_t stream) {
    const int G = a.num_heads / a.num_kv_heads;
    const int dpl = a.head_dim <= 64 ? 2 : (a.head_dim <= 128 ? 4 : 8);
    // query heads per CTA: the whole group up to 8 (4 with 8 dims per lane)
    const int gh = G == 1 ? 1 : (G <= 4 || dpl == 8 ? 4 : 8);
    dim3 grid((unsigned)a.total_q, (unsigned)(a.num_kv_heads * ((G + gh - 1) / gh)));
    const dim3 block(kWarps * 32);
#define PA_SIMT(D, H) attn_simt_kernel<T, FP8, D, H><<<grid, block, 0, stream>>>(a)
    if (dpl == 2) {
        if (gh == 1) PA_SIMT(2, 1);
        else if (gh == 4) PA_SIMT(2, 4);
        else PA_SIMT(2, 8);
    } else if (dpl == 4) {
        if (gh == 1) PA_SIMT(4, 1);
        else if (gh == 4) PA_SIMT(4, 4);
        else PA_SIMT(4, 8);
    } else {
        if (gh == 1) PA_SIMT(8, 1);
        else PA_SIMT(8, 4);
    }
#undef PA_SIMT
    return cudaGetLastError();
}

}  // namespace

bool attn_simt_supported(int dtype, int head_dim) {
    return (dtype >= 0 && dtype <= 2) && head_dim >= 1 && head_dim <= 32 * kMaxDimsPerLane;
}

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t stream) {
    if (a.total_q == 0) return cudaSuccess;
    if (a.kv_fp8) {
        switch (a.dtype) {
            case 0: return launch_typed<float, true>(a, stream);
            case 1: return launch_typed<__nv_bfloat16, true>(a, stream);
            default: return launch_typed<__half, true>(a, stream);
        }
    }
    switch (a.dtype) {
        case 0: return launch_typed<float, false>(a, stream);
        case 1: return launch_typed<__nv_bfloat16, false>(a, stream);
        default: return launch_typed<__half, false>(a, stream);
    }
}

}  // namespace pa
