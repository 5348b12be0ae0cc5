// pa_varlen_umma.cu -- the varlen prefill/decode mix on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), bf16/f16,
// head_dim 64 or 128, block_size 16.
//
// Same arithmetic as the handbook's paged_attention ("分页 KV Cache",
// §分页注意力): request i owns query rows cu[i] .. cu[i+1]-1, its new token j
// is at position L_i - n_i + j and (causal) sees keys 0..that position; query
// head h reads KV head h / G.
//
// A CTA takes one KV head and T = floor(128 / G) consecutive new tokens of one
// request, i.e. a 128-row tile of (token, group head) pairs -- the G heads
// share every K/V tile.  Roles:
//   warp 4              TMA: the Q tile once, then 64-key K and V tiles (four
//                       16-token blocks through the block table, staged in
//                       windows of 512 entries) into separate 2-slot K and V
//                       rings, so the next K tile loads as soon as its S is
//                       done, not after P V (two CTAs share an SM);
//   warp 5 (one lane)   issues tcgen05.mma: S = Q K^T (M 128, N 64, K = hd)
//                       into tensor memory, then O += P V (M 128, N hd, K 64)
//                       with V read MN-major; completion via tcgen05.commit;
//   warps 0-3           one query row per thread: read S from tensor memory,
//                       causal mask, exp2-domain online softmax, P (bf16/f16)
//                       written back to tensor memory as the A operand of
//                       P V; O is rescaled in tensor memory only when a row's
//                       running maximum grows by more than 2^8, and
//                       normalised and stored at the end.
// S(k+1) is issued as soon as the softmax warps have read S(k), so it runs
// under their exponentials.  V rows past the context are zeroed in shared
// memory before P V.  Every wait is bounded in time; on expiry the CTA sets a
// status bit, abandons the tile and still frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <string>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_umma_status;

constexpr int BS = 16;          // keys per group (one TMA box of 16 rows, or two of 8)
constexpr int BK = 64;          // keys per tile
constexpr int BPT = BK / BS;    // groups per key tile
constexpr int TM = 128;         // rows of the MMA tile
constexpr int R = 2;            // K/V stages
constexpr int NTHREADS = 192;   // 4 softmax warps + producer + MMA warp
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t S_COL = 0, P_COL = 64, O_COL = 128;  // S 64 fp32 cols, P 32 packed cols, O hd cols
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s
constexpr int kMaxSeqsSmem = 8192;
constexpr int kTableWindow = 512;  // block-table entries the producer stages at a time

struct UmParams {
    void* out;
    const int32_t* block_tables;
    int32_t max_blocks;
    const int32_t* seq_lens;
    const int32_t* cu;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t group;
    int32_t tokens_per_tile;  // T = floor(128 / group)
    int32_t block_size;       // tokens per pool block: 8, or a multiple of 16 up to 256
    int32_t causal;
    float scale_log2;
};

template <int HD>
struct UGeo {
    static constexpr int CH = HD / 64;          // 128-byte chunks per head row
    static constexpr int QCH = TM * 128;        // bytes of one chunk of the Q tile
    static constexpr int KCH = BK * 128;        // bytes of one chunk of a K (or V) tile
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = CH * QCH;
    static constexpr int TILE = CH * KCH;       // bytes of a K (or V) tile
    static constexpr int V_OFF = KV_OFF + R * TILE;
    static constexpr int BAR_OFF = V_OFF + R * TILE;
    // q_full, k_full[R], k_empty[R], v_full[R], v_empty[R], s_full, s_free, p_full, o_done
    static constexpr int NBAR = 1 + 4 * R + 4;
    static constexpr int TADDR_OFF = BAR_OFF + NBAR * 8;
    static constexpr int TBL_OFF = TADDR_OFF + 16;          // window of block-table entries
    static constexpr int CU_OFF = TBL_OFF + 2 * kTableWindow * 4;  // rows of each group's first and second box
};

template <int HD>
size_t um_smem_bytes(int num_seqs) {
    return 1024 + (size_t)UGeo<HD>::CU_OFF + (size_t)((num_seqs < kMaxSeqsSmem ? num_seqs : kMaxSeqsSmem) + 1) * 4;
}

template <typename T, int HD>
__global__ void __launch_bounds__(NTHREADS, 2)
    varlen_umma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const UmParams p) {
    using Gm = UGeo<HD>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + Gm::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = bars + 1 + R;
    uint64_t* v_full = bars + 1 + 2 * R;
    uint64_t* v_empty = bars + 1 + 3 * R;
    uint64_t* s_full = bars + 1 + 4 * R;
    uint64_t* s_free = s_full + 1;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_done = s_full + 3;
    volatile uint32_t* taddr_slot = reinterpret_cast<volatile uint32_t*>(base + Gm::TADDR_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + Gm::TADDR_OFF + 4);
    int32_t* cu_s = reinterpret_cast<int32_t*>(base + Gm::CU_OFF);
    int32_t* tbl_s = reinterpret_cast<int32_t*>(base + Gm::TBL_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.num_seqs, G = p.group, TT = p.tokens_per_tile;
    const int kvh = blockIdx.y;
    pdl_wait_primary();

    // ---- request and tile: request i owns tiles [floor(cu[i]/T) + i, floor(cu[i+1]/T) + i + 1)
    const bool cu_in_smem = S <= kMaxSeqsSmem;
    if (cu_in_smem)
        for (int i = threadIdx.x; i <= S; i += blockDim.x) cu_s[i] = p.cu[i];
    __syncthreads();
    auto cu_at = [&](int i) -> int { return cu_in_smem ? cu_s[i] : p.cu[i]; };
    auto tile0 = [&](int i) -> int64_t { return (int64_t)cu_at(i) / TT + i; };
    const int64_t bid = blockIdx.x;
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile0(mid) <= bid) lo = mid;
        else hi = mid - 1;
    }
    const int req = lo;
    const int q0 = cu_at(req), n_new = cu_at(req + 1) - q0;
    const int ntile = (n_new + TT - 1) / TT;
    const int64_t t_rel = bid - tile0(req);
    if (t_rel >= ntile) return;  // the spare tile of this request (uniform for the CTA)
    const int t0 = (ntile - 1 - (int)t_rel) * TT;  // last tiles first
    const int tn = min(TT, n_new - t0);
    const int L = p.seq_lens[req];
    const int first_pos = L - n_new;
    const int kv_end = p.causal ? first_pos + t0 + tn : L;
    const int nkt = (kv_end + BK - 1) / BK;
    const int nb_seq = (L + BS - 1) / BS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Gm::NBAR; ++i) mbar_init(&bars[i], (&bars[i] == s_free || &bars[i] == p_full) ? 4u : 1u);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(const_cast<uint32_t*>(taddr_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;
    const uint32_t s_base = smem_u32(base);

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_umma_status, kStatusTimeout);
    };

    if (warp == 4) {
        // ---------------- producer: the whole warp stages block-table
        // windows (one round trip per 128 tiles), lane 0 issues the TMA loads
        const uint64_t pol = l2_policy_evict_last();
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            mbar_arrive_expect_tx(q_full, (uint32_t)(Gm::CH * 128 * G * TT));
#pragma unroll
            for (int c = 0; c < Gm::CH; ++c)
                tma_load_3d(base + Gm::Q_OFF + c * Gm::QCH, &tmQ, q_full, 64 * c, kvh * G, q0 + t0, pol);
        }
        // pool row of every 16-key group this CTA reads (and of its second
        // 8-row box with 8-token blocks), staged a window at a time
        const int ngrp = min(nb_seq, nkt * BPT);
        const int32_t* table = p.block_tables + (int64_t)req * p.max_blocks;
        const int bsz = p.block_size;
        bool run = true;
        for (int w0 = 0; w0 < ngrp && run; w0 += kTableWindow) {
            const int wn = min(kTableWindow, ngrp - w0);
            for (int i = lane; i < wn; i += 32) {
                const int tok = (w0 + i) * BS;
                if (bsz == 8) {
                    const int32_t r1 = table[tok >> 3] * 8;
                    tbl_s[i] = r1;
                    tbl_s[kTableWindow + i] = tok + 8 < L ? table[(tok >> 3) + 1] * 8 : r1;
                } else {
                    tbl_s[i] = table[tok / bsz] * bsz + tok % bsz;
                }
            }
            __syncwarp();
            if (lane == 0) {
                const int kt_end = min(nkt, (w0 + wn + BPT - 1) / BPT);
                for (int kt = w0 / BPT; kt < kt_end; ++kt) {
                    if (*abort_flag) {
                        run = false;
                        break;
                    }
                    const int slot = kt % R;
                    const uint32_t par = ((uint32_t)(kt / R) & 1u) ^ 1u;
                    const int nvalid = min(BPT, nb_seq - kt * BPT);
                    const uint32_t bytes = (uint32_t)(nvalid * Gm::CH * BS * 128);
                    for (int half = 0; half < 2 && run; ++half) {  // K tile, then V tile
                        uint64_t* emp = half ? &v_empty[slot] : &k_empty[slot];
                        uint64_t* ful = half ? &v_full[slot] : &k_full[slot];
                        if (!mbar_wait_ns(emp, par, WAIT_NS)) {
                            fail();
                            run = false;
                            break;
                        }
                        uint8_t* st = base + (half ? Gm::V_OFF : Gm::KV_OFF) + slot * Gm::TILE;
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(ful, bytes);
                        for (int j = 0; j < nvalid; ++j) {  // groups past the context are never read
                            const int e = kt * BPT + j - w0;
                            const int row = tbl_s[e];
#pragma unroll
                            for (int c = 0; c < Gm::CH; ++c) {
                                uint8_t* dst = st + c * Gm::KCH + j * BS * 128;
                                if (bsz == 8) {  // two 8-row boxes, each a 1024-byte swizzle atom
                                    tma_load_3d(dst, half ? &tmV : &tmK, ful, 0, kvh * Gm::CH + c, row, pol);
                                    tma_load_3d(dst + 1024, half ? &tmV : &tmK, ful, 0, kvh * Gm::CH + c,
                                                tbl_s[kTableWindow + e], pol);
                                } else {
                                    tma_load_3d(dst, half ? &tmV : &tmK, ful, 0, kvh * Gm::CH + c, row, pol);
                                }
                            }
                        }
                    }
                    if (!run) break;
                }
            }
            run = __shfl_sync(0xffffffffu, run ? 1 : 0, 0) != 0;
            __syncwarp();
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idS = umma_idesc_f16(TM, BK, kBF16, false);
            const uint32_t idO = umma_idesc_f16(TM, HD, kBF16, true);
            const uint32_t q_s = s_base + Gm::Q_OFF;
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait_ns(&v_full[j % R], (uint32_t)(j / R) & 1u, WAIT_NS) ||
                    !mbar_wait_ns(p_full, (uint32_t)j & 1u, WAIT_NS))
                    return false;
                tc_fence_after();
                const uint32_t v_s = s_base + Gm::V_OFF + (j % R) * Gm::TILE;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t b = umma_sdesc_sw128(v_s + kk * 16 * 128, Gm::KCH, 1024);
                    umma_f16_ts(tmem + O_COL, tmem + P_COL + kk * 8, b, idO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(o_done);
                umma_commit(&v_empty[j % R]);
                return true;
            };
            bool ok = mbar_wait_ns(q_full, 0, WAIT_NS);
            for (int kt = 0; ok && kt < nkt && !*abort_flag; ++kt) {
                const int slot = kt % R;
                ok = mbar_wait_ns(&k_full[slot], (uint32_t)(kt / R) & 1u, WAIT_NS) &&
                     (kt == 0 || mbar_wait_ns(s_free, (uint32_t)(kt - 1) & 1u, WAIT_NS));
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_s = s_base + Gm::KV_OFF + slot * Gm::TILE;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const int c = kk >> 2, koff = (kk & 3) * 32;
                    const uint64_t a = umma_sdesc_sw128(q_s + c * Gm::QCH + koff, 16, 1024);
                    const uint64_t b = umma_sdesc_sw128(k_s + c * Gm::KCH + koff, 16, 1024);
                    umma_f16(tmem + S_COL, a, b, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(s_full);
                umma_commit(&k_empty[slot]);
                if (kt > 0) ok = issue_pv(kt - 1);
            }
            if (ok && !*abort_flag) ok = issue_pv(nkt - 1);
            if (!ok) fail();
        }
    } else {
        // ---------------- softmax + epilogue: one query row per thread
        const int m = threadIdx.x;
        const bool valid = m < tn * G;
        const int ti = valid ? m / G : 0, gh = valid ? m - (m / G) * G : 0;
        const int prow = p.causal ? first_pos + t0 + ti : L - 1;
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int kt = 0; kt < nkt; ++kt) {
            if (*abort_flag || !mbar_wait_ns(s_full, (uint32_t)kt & 1u, WAIT_NS)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float sv[64];
            {
                float a[32], b[32];
                tmem_ld32(t_lane + S_COL, a);
                tmem_ld32(t_lane + S_COL + 32, b);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    sv[j] = a[j];
                    sv[32 + j] = b[j];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);

            const int kbase = kt * BK;
            // Raw scores; the mask only applies on tiles that reach past the
            // row's last visible key (the causal diagonal or the context end).
            // Rows past the request's pairs hold no query: flat zero scores,
            // so they never force a rescale of the warp.
            float mx = -INFINITY;
            if (!valid) {
#pragma unroll
                for (int j = 0; j < 64; ++j) sv[j] = 0.f;
                mx = 0.f;
            } else if (kbase + BK - 1 > prow) {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const float x = kbase + j > prow ? -INFINITY : sv[j];
                    sv[j] = x;
                    mx = fmaxf(mx, x);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) mx = fmaxf(mx, sv[j]);
            }
            // exp2 domain: x = s * scale * log2(e); a positive scale keeps the
            // order, so the maximum is taken on raw scores and the scaling is
            // fused into the exponent's argument
            const float sl = p.scale_log2;
            float m_tile;
            if (sl > 0.f) {
                m_tile = mx * sl;
            } else {
                m_tile = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; ++j) m_tile = fmaxf(m_tile, sv[j] == -INFINITY ? -INFINITY : sv[j] * sl);
            }
            const float m_new = fmaxf(m_used, m_tile);
            const bool grow = (m_used == -INFINITY) || (m_new > m_used + 8.f);
            float alpha = 1.f;
            if (grow) {
                alpha = fast_exp2(m_used - m_new);
                m_used = m_new;
            }
            const float neg_m = -m_used;
            float sum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float a0 = sv[2 * j] == -INFINITY ? -INFINITY : fmaf(sv[2 * j], sl, neg_m);
                const float a1 = sv[2 * j + 1] == -INFINITY ? -INFINITY : fmaf(sv[2 * j + 1], sl, neg_m);
                const float e0 = fast_exp2(a0), e1 = fast_exp2(a1);
                sum += e0 + e1;
                pk[j] = pack2<T>(e0, e1);
            }
            l = l * alpha + sum;
            const bool rescale = __any_sync(0xffffffffu, grow && kt > 0);

            if (kt > 0) {  // P V of the previous tile must be done: P buffer and O are shared
                if (!mbar_wait_ns(o_done, (uint32_t)(kt - 1) & 1u, WAIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (rescale) {
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    float o[32];
                    tmem_ld32(t_lane + O_COL + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= alpha;
                    tmem_st32(t_lane + O_COL + 32 * c, o);
                }
                tmem_wait_st();
            }
            // keys at or past L hold no context: zero their V rows of this stage
            const int keep = L - kbase;
            if (keep < BK) {
                // this tile's V must have landed before its tail rows are cleared
                if (!mbar_wait_ns(&v_full[kt % R], (uint32_t)(kt / R) & 1u, WAIT_NS)) {
                    ok = false;
                    break;
                }
                uint8_t* v_t = base + Gm::V_OFF + (kt % R) * Gm::TILE;
                const int rows = BK - keep;
                for (int e = threadIdx.x; e < rows * Gm::CH * 8; e += 128) {
                    const int c = e / (rows * 8), rem = e - c * rows * 8, r = keep + rem / 8, q16 = rem & 7;
                    *reinterpret_cast<uint4*>(v_t + c * Gm::KCH + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            // P row: 64 keys packed two per column into tensor memory
            {
                float pf[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) pf[j] = __uint_as_float(pk[j]);
                tmem_st32(t_lane + P_COL, pf);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && !*abort_flag && mbar_wait_ns(o_done, (uint32_t)(nkt - 1) & 1u, WAIT_NS)) {
            tc_fence_after();
            const float inv = 1.f / l;
            T* orow = static_cast<T*>(p.out) +
                      ((int64_t)(q0 + t0 + ti) * p.num_heads + (int64_t)kvh * G + gh) * HD;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                float o[32];
                tmem_ld32(t_lane + O_COL + 32 * c, o);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int q16 = 0; q16 < 4; ++q16) {
                        uint4 v;
                        v.x = pack2<T>(o[8 * q16 + 0] * inv, o[8 * q16 + 1] * inv);
                        v.y = pack2<T>(o[8 * q16 + 2] * inv, o[8 * q16 + 3] * inv);
                        v.z = pack2<T>(o[8 * q16 + 4] * inv, o[8 * q16 + 5] * inv);
                        v.w = pack2<T>(o[8 * q16 + 6] * inv, o[8 * q16 + 7] * inv);
                        *reinterpret_cast<uint4*>(orow + 32 * c + 8 * q16) = v;
                    }
                }
            }
        } else if (!ok || *abort_flag) {
            fail();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 um_encode_fn() {
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

bool um_encode(CUtensorMap* m, const void* base, int dtype, const cuuint64_t dims[3], const cuuint64_t strides[2],
               const cuuint32_t box[3], std::string* err) {
    auto fn = um_encode_fn();
    if (!fn) {
        *err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
        return false;
    }
    return true;
}

template <typename T, int HD>
cudaError_t um_launch(const AttnArgs& a, int32_t num_blocks, std::string* err, cudaStream_t stream) {
    const int G = a.num_heads / a.num_kv_heads;
    const int TT = TM / G;
    CUtensorMap tmQ, tmK, tmV;
    {
        // q as (hd elements) x (Hq heads) x (total_q tokens); one box = 64
        // elements of the G heads of a KV head over T tokens
        cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)a.num_heads, (cuuint64_t)a.total_q};
        cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)a.num_heads * HD * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TT};
        if (!um_encode(&tmQ, a.q, a.dtype, dims, strides, box, err)) return cudaErrorInvalidValue;
    }
    {
        const int ch = HD / 64;
        cuuint64_t dims[3] = {64, (cuuint64_t)a.num_kv_heads * ch, (cuuint64_t)num_blocks * a.block_size};
        cuuint64_t strides[2] = {128, (cuuint64_t)a.num_kv_heads * HD * 2};
        cuuint32_t box[3] = {64, 1, (cuuint32_t)(a.block_size == 8 ? 8 : BS)};
        if (!um_encode(&tmK, a.k_cache, a.dtype, dims, strides, box, err) ||
            !um_encode(&tmV, a.v_cache, a.dtype, dims, strides, box, err))
            return cudaErrorInvalidValue;
    }
    UmParams p;
    p.out = a.out;
    p.block_tables = a.block_tables;
    p.max_blocks = a.max_blocks;
    p.seq_lens = a.seq_lens;
    p.cu = a.cu_seqlens_q;
    p.num_seqs = a.num_seqs;
    p.num_heads = a.num_heads;
    p.group = G;
    p.tokens_per_tile = TT;
    p.block_size = a.block_size;
    p.causal = a.causal;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const int64_t tiles = (int64_t)a.total_q / TT + a.num_seqs;
    const size_t smem = um_smem_bytes<HD>(a.num_seqs);
    cudaError_t e = cudaFuncSetAttribute(varlen_umma_kernel<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)a.num_kv_heads);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, varlen_umma_kernel<T, HD>, tmQ, tmK, tmV, p);
}

}  // namespace

bool varlen_umma_supported(int dtype, int head_dim, int block_size, int group) {
    return (dtype == 1 || dtype == 2) && (head_dim == 64 || head_dim == 128) &&
           (block_size == 8 || (block_size % BS == 0 && block_size <= 256)) && group >= 1 &&
           group <= TM;
}

cudaError_t launch_varlen_umma(const AttnArgs& a, int32_t num_blocks, std::string* err, cudaStream_t stream) {
    if (a.total_q == 0 || a.num_seqs == 0) return cudaSuccess;
    if (a.dtype == 1)
        return a.head_dim == 64 ? um_launch<__nv_bfloat16, 64>(a, num_blocks, err, stream)
                                : um_launch<__nv_bfloat16, 128>(a, num_blocks, err, stream);
    return a.head_dim == 64 ? um_launch<__half, 64>(a, num_blocks, err, stream)
                            : um_launch<__half, 128>(a, num_blocks, err, stream);
}

uint32_t varlen_umma_status(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_umma_status, sizeof(v));
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_umma_status, &z, sizeof(z));
    }
    return v;
}

}  // namespace pa
