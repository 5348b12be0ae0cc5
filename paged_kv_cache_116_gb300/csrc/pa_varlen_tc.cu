// pa_varlen_tc.cu -- the varlen prefill/decode mix on the tensor cores
// (bf16/f16, head_dim 64 or 128, block_size 16).
//
// What it computes is the handbook's paged_attention ("分页 KV Cache",
// §分页注意力): request i owns query rows cu[i] .. cu[i+1]-1, its new token j
// sits at position L_i - n_i + j and (causal) sees positions 0..that one,
// query head h reads KV head h / G.
//
// How:
//  * A CTA takes one KV head and a tile of 64 consecutive (query row, head
//    of the group) pairs of one request -- the request's n_i * G pairs in
//    row-major order -- so the G heads of a KV head share every K/V tile the
//    CTA loads, and a decode row (n_i = 1) is one tile.  Tiles are numbered
//    per request from floor(cu[i] * G / 64) + i, which needs no scan: one
//    spare tile per request at most, and it exits at once.  Within a request
//    the tiles run last-first, so the ones with the longest key ranges start
//    earliest.
//  * A producer warp walks the keys 64 at a time (four 16-token blocks read
//    through the block table) and loads K and V tiles with TMA
//    (cp.async.bulk.tensor, 128-byte swizzle) into a 3-stage ring guarded by
//    full/empty mbarriers.
//  * Four consumer warps each own 16 of the 64 pairs: S = Q K^T and
//    O += P V with mma.m16n8k16 (fp32 accumulation), an exp2-domain online
//    softmax per row, the causal limit applied per row, and V rows past the
//    context zeroed in the operand so unused slots never leak.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <string>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_varlen_status;

constexpr int BS = 16;        // tokens per block
constexpr int BK = 64;        // keys per tile
constexpr int BPT = BK / BS;  // blocks per key tile
constexpr int TM = 64;        // (row, head) pairs per CTA
constexpr int NC = 4;         // consumer warps (16 pairs each)
constexpr int kMaxSeqsSmem = 8192;
constexpr int kTableWindow = 512;  // block-table entries the producer stages at a time

struct VlParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    int32_t max_blocks;
    const int32_t* seq_lens;
    const int32_t* cu;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t group;
    int32_t causal;
    float scale_log2;
};

template <int HD>
struct VGeo {
    static constexpr int CH = HD * 2 / 128;  // 128-byte chunks per head row
    static constexpr int BLK = BS * 128;     // bytes of one chunk of one block (16 rows x 128 B)
    static constexpr int TILE = BK * HD * 2; // bytes of a K (or V) tile of 64 keys
    static constexpr int STAGE = 2 * TILE;
    static constexpr int KS = HD / 16;       // k-steps of Q K^T
    static constexpr int NO = HD / 8;        // n-tiles of O
    static constexpr int R = HD == 128 ? 3 : 4;
};

template <int HD>
constexpr size_t vl_smem_bytes(int num_seqs) {
    return 1024 + (size_t)VGeo<HD>::R * VGeo<HD>::STAGE + (size_t)VGeo<HD>::R * 16 + kTableWindow * 4 +
           (size_t)((num_seqs < kMaxSeqsSmem ? num_seqs : kMaxSeqsSmem) + 1) * 4;
}

// Smem address of element (key, dim) in a tile laid out as [chunk][block]
// [16 rows][128 B] with the 128-byte swizzle inside each 8-row group.
__device__ __forceinline__ uint32_t vswz(int key, int dstart) {
    const int c = dstart >> 6, j = (dstart & 63) >> 3, blk = key >> 4, row = key & 15;
    return (uint32_t)(((c * BPT + blk) * BS + row) * 128 + ((j ^ (row & 7)) << 4));
}

template <typename T, int HD>
__global__ void __launch_bounds__((NC + 1) * 32)
    varlen_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const VlParams p) {
    using Gm = VGeo<HD>;
    constexpr int R = Gm::R, KS = Gm::KS, NO = Gm::NO;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)R * Gm::STAGE);
    uint64_t* empty = full + R;
    int32_t* tbl_s = reinterpret_cast<int32_t*>(empty + R);
    int32_t* cu_s = tbl_s + kTableWindow;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.num_seqs, G = p.group;
    const int kvh = blockIdx.y;
    pdl_wait_primary();

    // ---- which request and tile: request i owns tiles [floor(cu[i]*G/TM) + i, floor(cu[i+1]*G/TM) + i + 1)
    const bool cu_in_smem = S <= kMaxSeqsSmem;
    if (cu_in_smem)
        for (int i = threadIdx.x; i <= S; i += blockDim.x) cu_s[i] = p.cu[i];
    __syncthreads();
    auto cu_at = [&](int i) -> int { return cu_in_smem ? cu_s[i] : p.cu[i]; };
    auto tile0 = [&](int i) -> int64_t { return (int64_t)cu_at(i) * G / TM + i; };
    const int64_t bid = blockIdx.x;
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile0(mid) <= bid) lo = mid;
        else hi = mid - 1;
    }
    const int req = lo;
    const int q0 = cu_at(req), n_new = cu_at(req + 1) - q0;
    const int pairs = n_new * G;
    const int ntile = (pairs + TM - 1) / TM;
    const int64_t t_rel = bid - tile0(req);
    if (t_rel >= ntile) return;  // the spare tile of this request
    const int tile = ntile - 1 - (int)t_rel;  // last tiles first
    const int m0 = tile * TM;
    const int L = p.seq_lens[req];
    const int first_pos = L - n_new;  // position of new token 0
    // key range of the CTA: up to the last row it holds
    const int last_pair = min(m0 + TM, pairs) - 1;
    const int kv_end = p.causal ? first_pos + last_pair / G + 1 : L;
    const int nkt = (kv_end + BK - 1) / BK;
    const int nb_seq = (L + BS - 1) / BS;
    const int32_t* table = p.block_tables + (int64_t)req * p.max_blocks;

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&empty[r], NC);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == NC) {
        // ---------------- producer: the whole warp stages block-table
        // windows (one round trip per 128 tiles), lane 0 issues the TMA loads
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
        }
        const uint64_t pol = l2_policy_evict_last();
        const int nblk = min(nb_seq, nkt * BPT);
        bool run = true;
        for (int w0 = 0; w0 < nblk && run; w0 += kTableWindow) {
            const int wn = min(kTableWindow, nblk - w0);
            for (int i = lane; i < wn; i += 32) tbl_s[i] = table[w0 + i];
            __syncwarp();
            if (lane == 0) {
                const int kt_end = min(nkt, (w0 + wn + BPT - 1) / BPT);
                for (int kt = w0 / BPT; kt < kt_end; ++kt) {
                    const int slot = kt % R;
                    if (!mbar_wait_bounded(&empty[slot], ((uint32_t)(kt / R) & 1u) ^ 1u, kMaxPolls)) {
                        atomicOr(&g_varlen_status, kStatusTimeout);
                        run = false;
                        break;
                    }
                    const int nvalid = min(BPT, nb_seq - kt * BPT);
                    uint8_t* dst = base + (size_t)slot * Gm::STAGE;
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(nvalid * 2 * Gm::CH * Gm::BLK));
                    for (int j = 0; j < nvalid; ++j) {  // blocks past the context are never read
                        const int row = tbl_s[kt * BPT + j - w0] * BS;
#pragma unroll
                        for (int c = 0; c < Gm::CH; ++c) {
                            const int off = (c * BPT + j) * Gm::BLK;
                            tma_load_3d(dst + off, &tmK, &full[slot], 0, kvh * Gm::CH + c, row, pol);
                            tma_load_3d(dst + Gm::TILE + off, &tmV, &full[slot], 0, kvh * Gm::CH + c, row, pol);
                        }
                    }
                }
            }
            run = __shfl_sync(0xffffffffu, run ? 1 : 0, 0) != 0;
            __syncwarp();
        }
        return;
    }

    // ---------------- consumers: warp owns pairs m0 + warp*16 .. +15
    const int g = lane >> 2, c4 = lane & 3;
    int prow[2];       // causal limit (last visible key) of the thread's two rows
    bool valid[2];
    const T* qrow[2];
    T* orow[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int m = m0 + warp * 16 + g + 8 * e;
        valid[e] = m < pairs;
        const int mm = valid[e] ? m : 0;
        const int r = mm / G, gh = mm - r * G;
        prow[e] = p.causal ? first_pos + r : L - 1;
        const int64_t off = ((int64_t)(q0 + r) * p.num_heads + (int64_t)kvh * G + gh) * HD;
        qrow[e] = static_cast<const T*>(p.q) + off;
        orow[e] = static_cast<T*>(p.out) + off;
    }
    uint32_t qa[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        const int d = kk * 16 + 2 * c4;
        qa[kk][0] = valid[0] ? *reinterpret_cast<const uint32_t*>(qrow[0] + d) : 0u;
        qa[kk][1] = valid[1] ? *reinterpret_cast<const uint32_t*>(qrow[1] + d) : 0u;
        qa[kk][2] = valid[0] ? *reinterpret_cast<const uint32_t*>(qrow[0] + d + 8) : 0u;
        qa[kk][3] = valid[1] ? *reinterpret_cast<const uint32_t*>(qrow[1] + d + 8) : 0u;
    }
    const int prow_min = __reduce_min_sync(0xffffffffu, min(prow[0], prow[1]));

    float o[NO][4];
#pragma unroll
    for (int nt = 0; nt < NO; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    // ldmatrix lane roles
    const int mi = lane >> 3, ri = lane & 7;
    const uint32_t st0 = smem_u32(base);
    bool ok = true;
    for (int kt = 0; kt < nkt; ++kt) {
        const int slot = kt % R;
        if (!mbar_wait_bounded(&full[slot], (uint32_t)(kt / R) & 1u, kMaxPolls)) {
            if (lane == 0) atomicOr(&g_varlen_status, kStatusTimeout);
            ok = false;
            break;
        }
        const uint32_t kt_s = st0 + (uint32_t)slot * Gm::STAGE, vt_s = kt_s + Gm::TILE;

        // S = Q K^T over 64 keys: 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {  // pairs of n-tiles: keys np*16 .. +15
                // matrices: (keys +0..7, dims +0..7), (keys +0..7, dims +8..15), (keys +8..15, ...), ...
                const int key = np * 16 + (mi >> 1) * 8 + ri, dst = kk * 16 + (mi & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kt_s + vswz(key, dst), b0, b1, b2, b3);
                mma16816<T>(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma16816<T>(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
            }
        }

        // mask (causal limit per row, context end) and online softmax
        const int kbase = kt * BK;
        const bool need_mask = kbase + BK - 1 > prow_min;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = kbase + nt * 8 + 2 * c4 + (e & 1);
                const int rr = e >> 1;
                float x = s[nt][e] * p.scale_log2;
                if (need_mask && key > prow[rr]) x = -INFINITY;
                s[nt][e] = x;
                mx[rr] = fmaxf(mx[rr], x);
            }
        float alpha[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
            const float mn = fmaxf(mrow[rr], mx[rr]);
            alpha[rr] = fast_exp2(mrow[rr] - mn);
            mrow[rr] = mn;
            lrow[rr] *= alpha[rr];
        }
#pragma unroll
        for (int nt = 0; nt < NO; ++nt) {
            o[nt][0] *= alpha[0];
            o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1];
            o[nt][3] *= alpha[1];
        }
        uint32_t pa_[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float p0 = fast_exp2(s[nt][0] - mrow[0]), p1 = fast_exp2(s[nt][1] - mrow[0]);
            const float p2 = fast_exp2(s[nt][2] - mrow[1]), p3 = fast_exp2(s[nt][3] - mrow[1]);
            lrow[0] += p0 + p1;
            lrow[1] += p2 + p3;
            const int kk = nt >> 1, hi_ = nt & 1;
            pa_[kk][hi_ * 2 + 0] = pack2<T>(p0, p1);
            pa_[kk][hi_ * 2 + 1] = pack2<T>(p2, p3);
        }

        // O += P V: 4 k-steps of 16 keys, NO n-tiles of 8 dims
        const int keys_left = L - kbase;  // keys at or past L hold no context
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            // A fragment order: (rows g, keys lo), (rows g+8, keys lo), (rows g, keys hi), (rows g+8, keys hi)
            const uint32_t a0 = pa_[kk][0], a1 = pa_[kk][1], a2 = pa_[kk][2], a3 = pa_[kk][3];
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (keys_left < BK) {
                const int k0 = kk * 16 + 2 * c4;
                mlo = (k0 < keys_left ? 0x0000ffffu : 0u) | (k0 + 1 < keys_left ? 0xffff0000u : 0u);
                mhi = (k0 + 8 < keys_left ? 0x0000ffffu : 0u) | (k0 + 9 < keys_left ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int np = 0; np < NO / 2; ++np) {  // pairs of dim n-tiles: dims np*16 .. +15
                // matrices: (keys +0..7, dims +0..7), (keys +8..15, dims +0..7), (keys +0..7, dims +8..15), ...
                const int key = kk * 16 + (mi & 1) * 8 + ri, dst = np * 16 + (mi >> 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vt_s + vswz(key, dst), b0, b1, b2, b3);
                b0 &= mlo;
                b1 &= mhi;
                b2 &= mlo;
                b3 &= mhi;
                mma16816<T>(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816<T>(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (!ok) return;

    // ---- normalise and store the thread's two rows
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 1);
        lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 2);
    }
    const float inv0 = 1.f / lrow[0], inv1 = 1.f / lrow[1];
#pragma unroll
    for (int nt = 0; nt < NO; ++nt) {
        const int d = nt * 8 + 2 * c4;
        if (valid[0]) *reinterpret_cast<uint32_t*>(orow[0] + d) = pack2<T>(o[nt][0] * inv0, o[nt][1] * inv0);
        if (valid[1]) *reinterpret_cast<uint32_t*>(orow[1] + d) = pack2<T>(o[nt][2] * inv1, o[nt][3] * inv1);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 vl_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool vl_kv_map(CUtensorMap* m, const void* cache, int dtype, int num_blocks, int num_kv_heads, int head_dim,
               std::string* err) {
    auto fn = vl_encode_fn();
    if (!fn) {
        *err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    const int ch = head_dim * 2 / 128;
    cuuint64_t dims[3] = {64, (cuuint64_t)num_kv_heads * ch, (cuuint64_t)num_blocks * BS};
    cuuint64_t strides[2] = {128, (cuuint64_t)num_kv_heads * head_dim * 2};
    cuuint32_t box[3] = {64, 1, BS};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
        return false;
    }
    return true;
}

template <typename T, int HD>
cudaError_t vl_launch(const AttnArgs& a, int32_t num_blocks, std::string* err, cudaStream_t stream) {
    CUtensorMap tmK, tmV;
    if (!vl_kv_map(&tmK, a.k_cache, a.dtype, num_blocks, a.num_kv_heads, HD, err) ||
        !vl_kv_map(&tmV, a.v_cache, a.dtype, num_blocks, a.num_kv_heads, HD, err))
        return cudaErrorInvalidValue;
    VlParams p;
    p.out = a.out;
    p.q = a.q;
    p.block_tables = a.block_tables;
    p.max_blocks = a.max_blocks;
    p.seq_lens = a.seq_lens;
    p.cu = a.cu_seqlens_q;
    p.num_seqs = a.num_seqs;
    p.num_heads = a.num_heads;
    p.group = a.num_heads / a.num_kv_heads;
    p.causal = a.causal;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const int64_t tiles = (int64_t)a.total_q * p.group / TM + a.num_seqs;
    const size_t smem = vl_smem_bytes<HD>(a.num_seqs);
    cudaError_t e = cudaFuncSetAttribute(varlen_tc_kernel<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)a.num_kv_heads);
    cfg.blockDim = dim3((NC + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, varlen_tc_kernel<T, HD>, tmK, tmV, p);
}

}  // namespace

bool varlen_tc_supported(int dtype, int head_dim, int block_size) {
    return (dtype == 1 || dtype == 2) && (head_dim == 64 || head_dim == 128) && block_size == BS;
}

cudaError_t launch_varlen_tc(const AttnArgs& a, int32_t num_blocks, std::string* err, cudaStream_t stream) {
    if (a.total_q == 0 || a.num_seqs == 0) return cudaSuccess;
    if (a.dtype == 1)
        return a.head_dim == 64 ? vl_launch<__nv_bfloat16, 64>(a, num_blocks, err, stream)
                                : vl_launch<__nv_bfloat16, 128>(a, num_blocks, err, stream);
    return a.head_dim == 64 ? vl_launch<__half, 64>(a, num_blocks, err, stream)
                            : vl_launch<__half, 128>(a, num_blocks, err, stream);
}

uint32_t varlen_tc_status(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_varlen_status, sizeof(v));
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_varlen_status, &z, sizeof(z));
    }
    return v;
}

}  // namespace pa
