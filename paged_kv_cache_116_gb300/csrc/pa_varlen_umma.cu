// pa_varlen_umma.cu -- the varlen prefill/decode mix on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), bf16/f16,
// head_dim 64, 128 or 256, block_size 8 or a multiple of 16 up to 256
// (head_dim 256: a multiple of 16).  At head_dim 256 a CTA takes one query
// tile instead of two (S and O use 384 of the 512 tensor-memory columns) and
// its K and V rings have one slot (Q, K and V tiles of 64 KB each), and
// decode rows take the prefill path.
//
// Same arithmetic as the handbook's paged_attention ("分页 KV Cache",
// §分页注意力): request i owns query rows cu[i] .. cu[i+1]-1, its new token j
// is at position L_i - n_i + j and (causal) sees keys 0..that position; query
// head h reads KV head h / G.
//
// A query tile is one KV head's G query heads over T = floor(128 / G)
// consecutive new tokens of one request: 128 (token, head) rows that share
// every K/V tile.  One CTA per SM takes two adjacent query tiles of one
// request (A, the later tokens, and B), so each K/V tile that crosses the
// L2 -> shared-memory path feeds two 128-row MMAs.  Roles (352 threads):
//   warps 0-3 / 4-7     softmax of tile A / tile B: one query row per
//                       thread; read S from tensor memory, causal mask,
//                       exp2-domain online softmax, P (bf16/f16) written
//                       back to tensor memory as the A operand of P V; O is
//                       rescaled in tensor memory only when a row's running
//                       maximum grows by more than 2^8, and normalised and
//                       stored at the end;
//   warp 8 / warp 9     TMA producers of the K / V tiles (128 keys = eight
//                       16-token groups through the block table, staged in
//                       windows of 512 entries), each into its own R-slot
//                       ring; a tile's boxes are issued by one lane each;
//   warp 10 (one lane)  issues tcgen05.mma as operands become ready:
//                       S = Q K^T (M 128, N 128, K = hd) per tile, then
//                       O += P V (M 128, N hd, K 128) with V read MN-major.
// 128-key tiles: an M128 x N64 MMA instruction takes as long as M128 x N128,
// so narrower S tiles would leave half the tensor pipe idle.
// Tensor memory (512 columns): tile X in columns 256 X .. 256 X + 255:
// S (128 fp32 columns), overwritten in place by P (bf16/f16, two per
// column), then O (hd columns).  The MMAs of one thread execute in issue
// order, so S_X(k+1), issued after P V_X(k), cannot overwrite P_X(k) before
// P V_X(k) has read it.  V rows past the context are zeroed in shared memory
// before P V.  Every wait is bounded in time; on expiry the CTA sets
// a status bit, abandons the tile and still frees its tensor memory.
//
// Decode rows (requests with one new token, at most 16 query heads per KV
// head) take another route: 128 MMA rows of which G are used, and three
// serial softmax / MMA hand-offs for a 300-token context, would hold an SM
// for ~14 us per row.  Instead one CTA takes eight such requests of a KV
// head, one warp each, and each warp streams its request's keys through its
// own two-stage TMA ring in 16-token tiles and works them on the CUDA-core
// tensor path: S^T = K Q^T with mma.m16n8k16 (the tile's 16 keys as M, the
// G query heads as N, so each K/V byte is read once for the group), an
// exp2-domain online softmax over the tile, P^T moved into B-fragment
// layout with movmatrix, O^T += V^T P^T in fp32 registers.
//
// The grid is [decode groups | prefill tile pairs | spare]: the decode
// CTAs go first, since each streams its requests at one warp's pace and,
// dispatched last, they were the tail of the launch.  With a workspace, a
// one-CTA plan kernel runs first and lists the prefill tile pairs longest
// first (bucketed by the number of 128-key tiles tile A reads) and the
// decode rows; the varlen kernel, its programmatic dependent, takes item
// blockIdx.x / Hkv for KV head blockIdx.x % Hkv, so the long pairs of every
// request and both heads start in the first waves and the short ones fill
// the tail.  Each CTA's output is independent of
// the others', so the order changes no result.  Without a workspace every
// CTA scans the requests' pair counts and decode flags (one packed
// exclusive prefix in shared memory) and finds its work, in request order,
// by binary search.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_umma_status;

constexpr int BS = 16;          // keys per group (one TMA box of 16 rows, or two of 8)
constexpr int BK = 128;         // keys per tile
constexpr int BPT = BK / BS;    // groups per key tile
constexpr int TM = 128;         // rows of the MMA tile
constexpr int NWARPS = 11;      // 2 x 4 softmax warps, K producer, V producer, MMA issuer
constexpr int NTHREADS = NWARPS * 32;
constexpr int W_KPROD = 8, W_VPROD = 9, W_MMA = 10;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0, P_COL = 0, O_COL = 128;  // within a tile's 256 columns (P over S)
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s
constexpr int kMaxSeqsSmem = 4096;
constexpr int kTableWindow = 512;  // block-table entries a producer stages at a time
constexpr int DG = 8;              // decode requests per decode CTA (one per warp)
constexpr int DR = 2;              // stages of a decode warp's ring
constexpr int kPairBits = 20;      // packed prefix: pairs in the low 20 bits, decode rank above
constexpr int kMaxDecodeGroupG = 16;
constexpr int kPairMask = (1 << kPairBits) - 1;
constexpr int kMaxPlanBuckets = 4096;  // 128-key tile counts the plan sorts apart (longer ones share the last)

struct UmParams {
    void* out;
    const void* q;
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
    // planned order (workspace given): plan[0] = prefill pairs, plan[1] =
    // decode rows; items[k] describes the k-th prefill CTA's tile pair in
    // full -- {request, tile A's first query row, its position, L with bit
    // 31 set when a tile B precedes it} -- so the CTA reads nothing else,
    // longest first; dec_req[r] = the request of decode rank r
    const int32_t* plan;
    const int4* items;
    const int32_t* dec_req;
    int32_t dec_ctas;  // decode-CTA slots per KV head, at the front of the grid
    // quantized cache (FP8 mode): fp32 scales [num_blocks, num_kv_heads, block_size]
    const float* k_scales;
    const float* v_scales;
};

// Head dims up to 128: two query tiles per CTA and two-slot K and V rings.
// Head dim 256: one query tile (S and O take 384 of the 512 tensor-memory
// columns) and one-slot rings (Q, K and V tiles of 64 KB each).
template <int HD>
struct UGeo {
    static constexpr int NQ = HD == 256 ? 1 : 2;  // query tiles per CTA (the pair width)
    static constexpr int RK = HD == 256 ? 1 : 2;  // K and V ring slots
    static constexpr int CH = HD / 64;          // 128-byte chunks per head row
    static constexpr int QCH = TM * 128;        // bytes of one chunk of a Q tile
    static constexpr int KCH = BK * 128;        // bytes of one chunk of a K (or V) tile
    static constexpr int QT = CH * QCH;         // bytes of a Q tile
    static constexpr int Q_OFF = 0;             // Q tiles A, B
    static constexpr int TILE = CH * KCH;       // bytes of a K (or V) tile
    static constexpr int K_OFF = NQ * QT;
    static constexpr int V_OFF = K_OFF + RK * TILE;
    static constexpr int BAR_OFF = V_OFF + RK * TILE;
    // q_full, k_full[R], k_empty[R], v_full[R], v_empty[R],
    // per tile: s_full, p_full, o_done; v_zeroed;
    // code cache only: k_conv[R], v_conv[R] (a slot's codes turned into
    // f16), q_conv (the Q tiles in f16)
    // (a decode CTA's warps use DR each of the same barriers)
    static constexpr int NBAR_PF = 1 + 4 * RK + 6 + 1 + 2 * RK + 1;
    static constexpr int NBAR = NBAR_PF > DG * DR ? NBAR_PF : DG * DR;
    static constexpr int TADDR_OFF = BAR_OFF + NBAR * 8;
    static constexpr int TBL_OFF = TADDR_OFF + 16;                 // two producers' table windows
    static constexpr int TBL_INTS = 2 * kTableWindow;              // rows of each group's first and second box
    // code cache: K then V scales per slot (targets of 16-byte-aligned bulk copies)
    static constexpr int SCL_OFF = (TBL_OFF + 2 * TBL_INTS * 4 + 127) / 128 * 128;
    // code cache: a prefill CTA's [2][R][BK] scales, or a decode CTA's [DG][DR][2][BS]
    static constexpr int SCL_BYTES = 2 * RK * BK * 4 > DG * DR * 2 * BS * 4 ? 2 * RK * BK * 4 : DG * DR * 2 * BS * 4;
    static constexpr int CU_OFF = SCL_OFF + SCL_BYTES;
};

static_assert(DG * DR <= UGeo<64>::NBAR, "a decode CTA's warps use the kernel's barriers");
static_assert(UGeo<128>::SCL_OFF % 128 == 0 && UGeo<64>::SCL_OFF % 128 == 0 && UGeo<256>::SCL_OFF % 128 == 0,
              "scale area aligned for bulk copies");
static_assert(UGeo<256>::CU_OFF + 1024 + (kMaxSeqsSmem + 1) * 4 <= 232448, "head_dim 256 fits in shared memory");
static_assert(DG * DR * 2 * BS * 64 * 2 <= UGeo<64>::BAR_OFF && DG * DR * 2 * BS * 128 * 2 <= UGeo<128>::BAR_OFF,
              "decode warps' stages fit below the barriers");

template <int HD>
size_t um_smem_bytes(int num_seqs) {
    return 1024 + (size_t)UGeo<HD>::CU_OFF + (size_t)((num_seqs < kMaxSeqsSmem ? num_seqs : kMaxSeqsSmem) + 1) * 4;
}

// One decode request (a single query at position L-1, which sees all L
// keys) for KV head kvh, worked by one warp: its G query heads' outputs.
// wst: the warp's DR stages of a 16-token K tile then V tile (1024-byte
// aligned, 128-byte swizzle as the tensor maps write them); wbar: DR
// mbarriers.  Returns false if a bounded wait ran out.
// FP8 (head_dim 128): the cache holds E4M3 codes with scales; each tile's
// codes land in the tile's second 128-byte chunk (where f16 row r of that
// chunk goes) and its 16 K and 16 V scales in `wscl` [DR][2][16]; once the
// tile has landed the warp turns it into f16 code x scale in place (V rows
// past the context become zeros), then the mma runs in f16.
template <typename T, int HD, int NT, bool FP8 = false>
__device__ __forceinline__ bool warp_decode(const CUtensorMap* tmK, const CUtensorMap* tmV, const UmParams& p,
                                            int req, int kvh, uint8_t* wst, uint64_t* wbar, float* wscl,
                                            int lane) {
    static_assert(!FP8 || HD == 128, "code tiles at head_dim 128");
    using MT = typename std::conditional<FP8, __half, T>::type;  // the mma operand type
    constexpr int CH = HD / 64, KS = HD / 16;
    constexpr int TILE = BS * HD * 2;  // bytes of a 16-token K (or V) tile
    constexpr int STAGE = 2 * TILE;
    const int G = p.group;
    const int Hkv = p.num_heads / G;
    const int L = p.seq_lens[req], qrow0 = p.cu[req];
    T* out = static_cast<T*>(p.out) + ((int64_t)qrow0 * p.num_heads + (int64_t)kvh * G) * HD;
    const int ntl = (L + BS - 1) / BS;
    if (ntl <= 0) {  // no context: a zero row
        for (int e = lane; e < G * HD; e += 32) out[e] = Elt<T>::from_f(0.f);
        return true;
    }
    const int32_t* table = p.block_tables + (int64_t)req * p.max_blocks;
    const int bsz = p.block_size;
    const uint64_t pol = l2_policy_evict_last();  // forked prompts are read by several requests
    // pool row of tile t's first token (and of its second 8-row half)
    auto entry = [&](int t, int32_t& row2) -> int32_t {
        row2 = 0;
        if (t >= ntl) return 0;
        const int tok = t * BS;
        if (bsz == 8) {
            const int32_t r1 = table[tok >> 3] * 8;
            row2 = tok + 8 < L ? table[(tok >> 3) + 1] * 8 : r1;
            return r1;
        }
        return table[tok / bsz] * bsz + tok % bsz;
    };
    int32_t trow2, trow = entry(lane, trow2);  // lane i: tile 32 win + i
    int win = 0;
    const int halves = bsz == 8 ? 2 : 1;
    const int nbox = FP8 ? 4 * halves : CH * 2 * halves;  // FP8: K, V code boxes and K, V scale copies
    auto issue = [&](int t) {
        if ((t >> 5) != win) {
            win = t >> 5;
            trow = entry(32 * win + lane, trow2);
        }
        const int slot = t % DR;
        const int32_t row = __shfl_sync(0xffffffffu, trow, t & 31), row2 = __shfl_sync(0xffffffffu, trow2, t & 31);
        if (lane == 0) mbar_arrive_expect_tx(&wbar[slot], FP8 ? (uint32_t)(2 * BS * (128 + 4)) : (uint32_t)(2 * TILE));
        fence_proxy_async_smem();  // this slot's previous tile was read by ldmatrix
        if (lane < nbox) {
            if constexpr (FP8) {
                const int hf = lane % halves, kind = lane / halves;  // 0 K codes, 1 V codes, 2 K scales, 3 V scales
                const int is_v = kind & 1;
                const int32_t r = hf ? row2 : row;
                if (kind < 2) {
                    tma_load_3d(wst + slot * STAGE + is_v * TILE + BS * 128 + hf * 1024, is_v ? tmV : tmK,
                                &wbar[slot], 0, kvh, r, pol);
                } else {
                    const int64_t si = (int64_t)(r / bsz) * Hkv * bsz + (int64_t)kvh * bsz + r % bsz;
                    bulk_g2s(wscl + (slot * 2 + is_v) * BS + hf * 8, (is_v ? p.v_scales : p.k_scales) + si,
                             (uint32_t)(BS * 4 / halves), &wbar[slot]);
                }
            } else {
                const int hf = lane % halves, c = (lane / halves) % CH, is_v = lane / (halves * CH);
                uint8_t* dst = wst + slot * STAGE + is_v * TILE + c * BS * 128 + hf * 1024;
                tma_load_3d(dst, is_v ? tmV : tmK, &wbar[slot], 0, kvh * CH + c, hf ? row2 : row, pol);
            }
        }
    };
    int ip = 0;
    for (; ip < DR && ip < ntl; ++ip) issue(ip);

    const int g = lane >> 2, c4 = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    const int k_tok = (mi & 1) * 8 + ri, k_dof = (mi >> 1) * 8;  // ldmatrix roles (K, non-transposed)
    const int v_tok = (mi >> 1) * 8 + ri, v_dof = (mi & 1) * 8;  // (V^T, transposed)
    auto swz = [](int tok, int dstart) -> uint32_t {
        const int c = dstart >> 6, j = (dstart & 63) >> 3;
        return (uint32_t)(c * BS * 128 + tok * 128 + ((j ^ (tok & 7)) << 4));
    };
    uint32_t qb[KS][NT][2];
    const T* qbase = static_cast<const T*>(p.q) + ((int64_t)qrow0 * p.num_heads + (int64_t)kvh * G) * HD;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = nt * 8 + g;
            if (hh < G) {
                const T* qp = qbase + (int64_t)hh * HD + kk * 16 + 2 * c4;
                qb[kk][nt][0] = *reinterpret_cast<const uint32_t*>(qp);
                qb[kk][nt][1] = *reinterpret_cast<const uint32_t*>(qp + 8);
                if (FP8 && !std::is_same<T, __half>::value) {  // the mma runs in f16
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const T* x = reinterpret_cast<const T*>(&qb[kk][nt][e]);
                        qb[kk][nt][e] = pack2<__half>(Elt<T>::to_f(x[0]), Elt<T>::to_f(x[1]));
                    }
                }
            } else {
                qb[kk][nt][0] = qb[kk][nt][1] = 0u;
            }
        }
    float acc[KS][NT][4], mrow[NT][2], lrow[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mrow[nt][0] = mrow[nt][1] = -INFINITY;
        lrow[nt][0] = lrow[nt][1] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) acc[kk][nt][0] = acc[kk][nt][1] = acc[kk][nt][2] = acc[kk][nt][3] = 0.f;
    }
    const float sl = p.scale_log2;
    const uint32_t st0 = smem_u32(wst);
    for (int t = 0; t < ntl; ++t) {
        const int slot = t % DR;
        if (!mbar_wait_ns(&wbar[slot], (uint32_t)(t / DR) & 1u, WAIT_NS)) {
            for (int u = t + 1; u < ip; ++u) mbar_wait_ns(&wbar[u % DR], (uint32_t)(u / DR) & 1u, WAIT_NS);
            return false;
        }
        const uint32_t kt = st0 + (uint32_t)slot * STAGE, vt = kt + TILE;
        const int valid = min(BS, L - t * BS);
        if constexpr (FP8) {
            // codes -> f16 (x scale) in place: lane (row lane & 15, half
            // lane >> 4) reads its row's 64 codes, then the warp writes
            uint8_t* tk = wst + (size_t)slot * STAGE;
            const int r = lane & 15, hh = lane >> 4;
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {  // K tile, then V tile
                uint4 c[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    c[j] = *reinterpret_cast<const uint4*>(tk + kv * TILE + BS * 128 + r * 128 +
                                                           (((4 * hh + j) ^ (r & 7)) << 4));
                __syncwarp();  // every lane holds its codes before any row is rewritten
                const bool zero = kv == 1 && r >= valid;
                const __half2 hs = __float2half2_rn(zero ? 0.f : wscl[(slot * 2 + kv) * BS + r]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {  // codes 64 hh + 16 j .. +15 -> f16 pieces 8 hh + 2 j, +1
                    const uint32_t w[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
                    uint32_t h[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t lo, hi;
                        e4m3x4_to_f16x2x2(w[u], lo, hi);
                        __half2 a, b;
                        memcpy(&a, &lo, 4);
                        memcpy(&b, &hi, 4);
                        a = zero ? __float2half2_rn(0.f) : __hmul2(a, hs);
                        b = zero ? __float2half2_rn(0.f) : __hmul2(b, hs);
                        memcpy(&h[2 * u], &a, 4);
                        memcpy(&h[2 * u + 1], &b, 4);
                    }
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int pj = 2 * j + half;  // piece within chunk hh
                        *reinterpret_cast<uint4*>(tk + kv * TILE + hh * BS * 128 + r * 128 + ((pj ^ (r & 7)) << 4)) =
                            make_uint4(h[4 * half], h[4 * half + 1], h[4 * half + 2], h[4 * half + 3]);
                    }
                }
                __syncwarp();
            }
        }
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kt + swz(k_tok, kk * 16 + k_dof), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816<MT>(sc[nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
        }
        const bool ok0 = g < valid, ok1 = g + 8 < valid;
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float x0 = ok0 ? sc[nt][0] * sl : -INFINITY, x1 = ok0 ? sc[nt][1] * sl : -INFINITY;
            const float x2 = ok1 ? sc[nt][2] * sl : -INFINITY, x3 = ok1 ? sc[nt][3] * sl : -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(mrow[nt][0], mx0), mn1 = fmaxf(mrow[nt][1], mx1);
            const float al0 = fast_exp2(mrow[nt][0] - mn0), al1 = fast_exp2(mrow[nt][1] - mn1);
            mrow[nt][0] = mn0;
            mrow[nt][1] = mn1;
            const float p0 = fast_exp2(x0 - mn0), p1 = fast_exp2(x1 - mn1);
            const float p2 = fast_exp2(x2 - mn0), p3 = fast_exp2(x3 - mn1);
            lrow[nt][0] = fmaf(lrow[nt][0], al0, p0 + p2);
            lrow[nt][1] = fmaf(lrow[nt][1], al1, p1 + p3);
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    acc[mt][nt][0] *= al0;
                    acc[mt][nt][1] *= al1;
                    acc[mt][nt][2] *= al0;
                    acc[mt][nt][3] *= al1;
                }
            }
            pb[nt][0] = movm_t(pack2<MT>(p0, p1));
            pb[nt][1] = movm_t(pack2<MT>(p2, p3));
        }
        // V rows past the context may hold anything: their operand lanes are zeroed
        uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
        if (valid < BS) {
            m01 = (2 * c4 < valid ? 0x0000ffffu : 0u) | (2 * c4 + 1 < valid ? 0xffff0000u : 0u);
            m23 = (2 * c4 + 8 < valid ? 0x0000ffffu : 0u) | (2 * c4 + 9 < valid ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vt + swz(v_tok, mt * 16 + v_dof), a0, a1, a2, a3);
            a0 &= m01;
            a1 &= m01;
            a2 &= m23;
            a3 &= m23;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816<MT>(acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
        }
        __syncwarp();
        if (ip < ntl) issue(ip++);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float l = lrow[nt][e];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const int hh = nt * 8 + 2 * c4 + e;
            if (hh < G) {
                const float inv = 1.f / l;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    out[hh * HD + mt * 16 + g] = Elt<T>::from_f(acc[mt][nt][e] * inv);
                    out[hh * HD + mt * 16 + g + 8] = Elt<T>::from_f(acc[mt][nt][2 + e] * inv);
                }
            }
        }
    return true;
}

// Code cache (FP8 mode, head_dim 128): a slot's 128 rows of 128 E4M3 codes,
// landed by TMA in the slot's second 128-byte chunk (row r at the offset of
// f16 row r of that chunk, same swizzle), become f16 values code x scale in
// both chunks, in place: each lane reads a row's 128 codes before writing
// that row.  Rows at or past `keep` (no context) are written as zeros when
// `zero_tail` (V: P is 0 there but a code may be NaN).
__device__ __forceinline__ void dequant_tile_in_place(uint8_t* slot, const float* scl, int keep, bool zero_tail,
                                                      int lane) {
    constexpr int KCH = BK * 128;
#pragma unroll 1
    for (int r = lane; r < BK; r += 32) {
        uint8_t* row1 = slot + KCH + r * 128;
        uint4 c[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] = *reinterpret_cast<const uint4*>(row1 + ((j ^ (r & 7)) << 4));
        const bool zero = zero_tail && r >= keep;
        const __half2 hs = __float2half2_rn(zero ? 0.f : scl[r]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // codes 16j .. 16j+15 -> f16 pieces 2j, 2j+1
            const uint32_t w[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
            uint32_t h[8];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                uint32_t lo, hi;
                e4m3x4_to_f16x2x2(w[t], lo, hi);
                __half2 a, b;
                memcpy(&a, &lo, 4);
                memcpy(&b, &hi, 4);
                a = zero ? __float2half2_rn(0.f) : __hmul2(a, hs);
                b = zero ? __float2half2_rn(0.f) : __hmul2(b, hs);
                memcpy(&h[2 * t], &a, 4);
                memcpy(&h[2 * t + 1], &b, 4);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int pc = 2 * j + half, ch = pc >> 3, pj = pc & 7;
                *reinterpret_cast<uint4*>(slot + ch * KCH + r * 128 + ((pj ^ (r & 7)) << 4)) =
                    make_uint4(h[4 * half], h[4 * half + 1], h[4 * half + 2], h[4 * half + 3]);
            }
        }
    }
}

template <typename T, int HD, bool FP8>
__global__ void __launch_bounds__(NTHREADS, 1)
    varlen_umma_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const UmParams p) {
    using Gm = UGeo<HD>;
    static_assert(!FP8 || HD == 128, "the code cache is read at head_dim 128");
    constexpr int R = Gm::RK;   // K and V ring slots at this head dim
    constexpr int PW = Gm::NQ;  // query tiles per CTA (2: a tile pair; 1: one tile)
    // the MMA operand type: the query type, or f16 over a code cache
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value && !FP8;
    using PT = typename std::conditional<FP8, __half, T>::type;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + Gm::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = bars + 1 + R;
    uint64_t* v_full = bars + 1 + 2 * R;
    uint64_t* v_empty = bars + 1 + 3 * R;
    uint64_t* tb = bars + 1 + 4 * R;  // per tile X: tb[3X] s_full, +1 p_full, +2 o_done
    uint64_t* v_zeroed = tb + 6;
    uint64_t* k_conv = v_zeroed + 1;
    uint64_t* v_conv = k_conv + R;
    uint64_t* q_conv = v_conv + R;
    float* scl_s = reinterpret_cast<float*>(base + Gm::SCL_OFF);  // [2][R][BK]: K, then V scales
    volatile uint32_t* taddr_slot = reinterpret_cast<volatile uint32_t*>(base + Gm::TADDR_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + Gm::TADDR_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.num_seqs, G = p.group, TT = p.tokens_per_tile;
    const bool planned = p.plan != nullptr;
    const int Hkv = p.num_heads / G;
    const int kvh = planned ? (int)(blockIdx.x % Hkv) : (int)blockIdx.y;
    // the tensor maps are kernel parameters: their descriptors are fetched
    // while this grid waits for the previous kernel (a first TMA through a
    // descriptor not yet fetched stalls its issuing thread)
    if (threadIdx.x == 32 * W_KPROD) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    pdl_wait_primary();

    // ---- work of this CTA.  Per request: its tile pairs (ceil(n / 2T); none
    // for a decode row taken by a decode CTA) and whether it is such a
    // decode row; one packed exclusive prefix of both over the requests.
    int32_t* pref = reinterpret_cast<int32_t*>(base + Gm::CU_OFF);  // [S + 1]
    const bool dec_route = G <= kMaxDecodeGroupG && HD <= 128;
    int64_t bid = blockIdx.x;
    int n_pairs, n_dec;
    int4 item = make_int4(0, 0, 0, 0);
    if (planned) {
        bid = blockIdx.x / Hkv;
        // a prefill slot's item is read with the plan's counts, not after
        // them: slots past the pairs read an unused entry (the item array
        // holds one per slot) and return below
        if (bid >= p.dec_ctas) item = __ldcg(p.items + (bid - p.dec_ctas));
        n_pairs = __ldcg(p.plan);
        n_dec = __ldcg(p.plan + 1);
    } else {
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        const int n = p.cu[i + 1] - p.cu[i];
        const bool dec = dec_route && n == 1;
        pref[i + 1] = dec ? (1 << kPairBits) : (n + PW * TT - 1) / (PW * TT);
    }
    if (threadIdx.x == 0) pref[0] = 0;
    __syncthreads();
    if (warp == 0) {
        const int per = (S + 31) / 32;
        const int lo = 1 + lane * per, hi = min(S + 1, lo + per);
        int sum = 0;
        for (int i = lo; i < hi; ++i) sum += pref[i];
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - sum;
        for (int i = lo; i < hi; ++i) {
            run += pref[i];
            pref[i] = run;
        }
    }
    __syncthreads();
    n_pairs = pref[S] & kPairMask;
    n_dec = pref[S] >> kPairBits;
    }
    if (bid < p.dec_ctas) {
        // ---- a decode CTA (or a spare one): decode rows of ranks DG d .. DG d + 7.
        // They lead the grid: each streams its requests' keys at one warp's
        // pace and would otherwise be the tail of the launch.
        const int64_t d = bid;
        if (d * DG >= n_dec) return;  // spare (uniform for the CTA)
        if (threadIdx.x == 0) {
            for (int w = 0; w < DG * DR; ++w) mbar_init(&bars[w], 1u);
            mbar_fence_init();
        }
        __syncthreads();
        const int rank = (int)(d * DG) + warp;
        if (warp >= DG || rank >= n_dec) return;
        int lo = 0;
        if (planned) {
            lo = __ldcg(p.dec_req + rank);
        } else {
            // the request with exactly `rank` decode rows before it and one more after it
            int hi = S - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if ((pref[mid + 1] >> kPairBits) > rank) hi = mid;
                else lo = mid + 1;
            }
        }
        if constexpr (HD <= 128) {  // (no decode CTAs at head_dim 256: dec_ctas is 0 there)
            constexpr int kStage = 2 * BS * HD * 2;
            uint8_t* wst = base + (size_t)warp * DR * kStage;
            float* wscl = scl_s + warp * DR * 2 * BS;  // FP8: this warp's [DR][2][16] scales
            const bool ok = G <= 8
                                ? warp_decode<T, HD, 1, FP8>(&tmK, &tmV, p, lo, kvh, wst, bars + warp * DR, wscl, lane)
                                : warp_decode<T, HD, 2, FP8>(&tmK, &tmV, p, lo, kvh, wst, bars + warp * DR, wscl, lane);
            if (!ok && lane == 0) atomicOr(&g_umma_status, kStatusTimeout);
        }
        return;
    }
    bid -= p.dec_ctas;
    if (bid >= n_pairs) return;  // spare (uniform for the CTA)
    // ---- a prefill CTA: tile pair p_rel of request req.  Per tile x (A the
    // later tokens, B the tile before it, if any): its first query row qrx,
    // the position of its first token psx, and its rows tnx.
    int req, L, ntiles, qrx[2], psx[2], tnx[2], nktx[2];
    if (planned) {
        const int4 it = item;
        req = it.x;
        L = it.w & 0x7fffffff;
        ntiles = it.w < 0 ? 2 : 1;
        qrx[0] = it.y;
        psx[0] = it.z;
        tnx[0] = min(TT, L - it.z);  // tile A ends at the request's last token or is full
        qrx[1] = it.y - TT;
        psx[1] = it.z - TT;
        tnx[1] = ntiles == 2 ? TT : 0;
    } else {
        int lo = 0, hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((pref[mid] & kPairMask) <= bid) lo = mid;
            else hi = mid - 1;
        }
        req = lo;
        const int p_rel = (int)(bid - (pref[req] & kPairMask));
        const int q0 = p.cu[req], n_new = p.cu[req + 1] - q0;
        L = p.seq_lens[req];
        // tile A = the later tokens (last pairs first); tile B the tile before it, if any
        const int tile_a = (n_new + TT - 1) / TT - 1 - PW * p_rel;
        ntiles = PW == 2 && tile_a >= 1 ? 2 : 1;
        for (int x = 0; x < 2; ++x) {
            const int t = tile_a - x, t0 = t >= 0 ? t * TT : 0;
            qrx[x] = q0 + t0;
            psx[x] = L - n_new + t0;
            tnx[x] = t >= 0 ? min(TT, n_new - t0) : 0;
        }
    }
    const int nb_seq = (L + BS - 1) / BS;
    for (int x = 0; x < 2; ++x) {
        const int kv_end = p.causal ? psx[x] + tnx[x] : L;
        nktx[x] = x < ntiles ? (kv_end + BK - 1) / BK : 0;
    }
    const int nkt = nktx[0];  // tile A reaches at least as far as tile B
    const int klast = (L - 1) / BK;  // the key tile holding the context end

    if (threadIdx.x == 0) {
        for (int i = 0; i < Gm::NBAR; ++i) mbar_init(&bars[i], 1u);
        for (int x = 0; x < 2; ++x) mbar_init(&tb[3 * x + 1], 4u);  // p_full: one arrival per softmax warp
        mbar_init(v_zeroed, 4u);
        mbar_init(q_conv, 8u);  // one arrival per softmax warp
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(const_cast<uint32_t*>(taddr_slot), TMEM_COLS);
        tmem_relinquish();
    }
    {
        // Q rows past the G x T (token, head) pairs get no TMA data: zero
        // them so their scores are finite and their (never stored) rows
        // take the same unmasked path as the rest of their warp
        const int pad = TM - G * TT, per_tile = Gm::CH * pad * 8;
        for (int e = threadIdx.x; e < PW * per_tile; e += NTHREADS) {
            const int x = e / per_tile, r0 = e - x * per_tile, c = r0 / (pad * 8), r = r0 - c * pad * 8;
            *reinterpret_cast<uint4*>(base + Gm::Q_OFF + x * Gm::QT + c * Gm::QCH + (G * TT + r / 8) * 128 +
                                      (r & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
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

    if (warp == W_KPROD || warp == W_VPROD) {
        // ---------------- producers: each stages its own block-table
        // windows; lane 0 waits for the next free slot of its ring, then the
        // tile's boxes are issued by one lane each in one instruction (a
        // single thread's TMA issue rate, not bandwidth, would bound the
        // load otherwise)
        const int is_v = warp == W_VPROD;
        const uint64_t pol = l2_policy_evict_last();
        const CUtensorMap* tm = is_v ? &tmV : &tmK;
        uint64_t* fulls = is_v ? v_full : k_full;
        uint64_t* emps = is_v ? v_empty : k_empty;
        int32_t* tbl_s = reinterpret_cast<int32_t*>(base + Gm::TBL_OFF) + is_v * Gm::TBL_INTS;
        if (lane == 0) {
            if (!is_v) {
                mbar_arrive_expect_tx(q_full, (uint32_t)(ntiles * Gm::CH * 128 * G * TT));
                for (int x = 0; x < ntiles; ++x)
#pragma unroll
                    for (int c = 0; c < Gm::CH; ++c)
                        tma_load_3d(base + Gm::Q_OFF + x * Gm::QT + c * Gm::QCH, &tmQ, q_full, 64 * c, kvh * G,
                                    qrx[x], pol);
            }
        }
        const int ngrp = min(nb_seq, nkt * BPT);
        const int32_t* table = p.block_tables + (int64_t)req * p.max_blocks;
        const int bsz = p.block_size;
        const int halves = bsz == 8 ? 2 : 1;
        // lanes per 16-token group: a box per chunk (16-bit) or a code box
        // and a scale copy (code cache), each per 8-row half with 8-token blocks
        const int per_group = (FP8 ? 2 : Gm::CH) * halves;
        const float* scales = is_v ? p.v_scales : p.k_scales;
        uint64_t* convs = is_v ? v_conv : k_conv;
        bool run = true;
        // code cache: a tile is turned into f16 while the next one loads
        int pending = -1;
        auto convert = [&](int t) -> bool {
            const int sl = t % R;
            if (!mbar_wait_ns(&fulls[sl], (uint32_t)(t / R) & 1u, WAIT_NS) || *abort_flag) return false;
            dequant_tile_in_place(base + (is_v ? Gm::V_OFF : Gm::K_OFF) + sl * Gm::TILE,
                                  scl_s + (is_v * R + sl) * BK, L - t * BK, is_v != 0, lane);
            fence_proxy_async_smem();  // the MMAs read these values through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&convs[sl]);
            return true;
        };
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
            const int kt_end = min(nkt, (w0 + wn + BPT - 1) / BPT);
            for (int kt = w0 / BPT; kt < kt_end && run; ++kt) {
                const int slot = kt % R;
                int ready = 0;
                if (lane == 0) {
                    ready = mbar_wait_ns(&emps[slot], ((uint32_t)(kt / R) & 1u) ^ 1u, WAIT_NS) && !*abort_flag;
                    if (!ready) fail();
                }
                if (!__shfl_sync(0xffffffffu, ready, 0)) {
                    run = false;
                    break;
                }
                const int nvalid = min(BPT, nb_seq - kt * BPT);
                uint8_t* st = base + (is_v ? Gm::V_OFF : Gm::K_OFF) + slot * Gm::TILE;
                if (lane == 0) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(&fulls[slot], FP8 ? (uint32_t)(nvalid * BS * (128 + 4))
                                                            : (uint32_t)(nvalid * Gm::CH * BS * 128));
                }
                __syncwarp();
                // lane = (group j, chunk c[, 8-row half]); groups past the context are never read
                if (lane < nvalid * per_group) {
                    const int j = lane / per_group, r = lane - j * per_group;
                    if constexpr (FP8) {
                        // r < halves: the group's code rows (into the slot's second
                        // chunk, where f16 row j*16+.. will be); else its scales
                        const int h8 = r % halves;
                        const int e = kt * BPT + j - w0;
                        const int row = h8 ? tbl_s[kTableWindow + e] : tbl_s[e];
                        if (r < halves) {
                            tma_load_3d(st + Gm::KCH + j * BS * 128 + h8 * 1024, tm, &fulls[slot], 0, kvh, row, pol);
                        } else {
                            const int64_t si = (int64_t)(row / bsz) * Hkv * bsz + (int64_t)kvh * bsz + row % bsz;
                            bulk_g2s(scl_s + (is_v * R + slot) * BK + j * BS + h8 * 8, scales + si,
                                     (uint32_t)(BS * 4 / halves), &fulls[slot]);
                        }
                    } else {
                        const int c = bsz == 8 ? (r >> 1) : r, h8 = bsz == 8 ? (r & 1) : 0;
                        const int e = kt * BPT + j - w0;
                        const int row = h8 ? tbl_s[kTableWindow + e] : tbl_s[e];
                        tma_load_3d(st + c * Gm::KCH + j * BS * 128 + h8 * 1024, tm, &fulls[slot], 0,
                                    kvh * Gm::CH + c, row, pol);
                    }
                }
                if constexpr (FP8) {
                    if (pending >= 0 && !convert(pending)) {
                        if (lane == 0) fail();
                        run = false;
                        break;
                    }
                    pending = kt;
                }
            }
            __syncwarp();
        }
        if constexpr (FP8) {
            if (run && pending >= 0 && !convert(pending) && lane == 0) fail();
        }
    } else if (warp == W_MMA) {
        // ---------------- MMA issuer, in a fixed staggered order:
        //   S_A(0) S_B(0) | P V_A(k) S_A(k+1) P V_B(k) S_B(k+1) | ...
        // so tile A's softmax runs while tile B's MMAs execute and the
        // other way round.  S_X(k+1) follows P V_X(k) in issue order, which
        // is what lets S overwrite P in place.  A K (V) slot is released
        // after the last S (P V) that reads it.
        if (lane == 0) {
            const uint32_t idS = umma_idesc_f16(TM, BK, kBF16, false);
            const uint32_t idO = umma_idesc_f16(TM, HD, kBF16, true);
            const int nka = nktx[0], nkb = nktx[1];
            auto issue_s = [&](int x, int k) {
                const uint32_t k_s = s_base + Gm::K_OFF + (k % R) * Gm::TILE;
                const uint32_t q_s = s_base + Gm::Q_OFF + x * Gm::QT;
                const uint32_t d = tmem + 256u * x + S_COL;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const int c = kk >> 2, koff = (kk & 3) * 32;
                    const uint64_t qa = umma_sdesc_sw128(q_s + c * Gm::QCH + koff, 16, 1024);
                    const uint64_t kb = umma_sdesc_sw128(k_s + c * Gm::KCH + koff, 16, 1024);
                    umma_f16(d, qa, kb, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&tb[3 * x]);
                if (x == 1 || k >= nkb) umma_commit(&k_empty[k % R]);  // last reader of K(k)
            };
            auto issue_pv = [&](int x, int j) {
                const uint32_t v_s = s_base + Gm::V_OFF + (j % R) * Gm::TILE;
                const uint32_t a_t = tmem + 256u * x + P_COL;
                const uint32_t d = tmem + 256u * x + O_COL;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t vb = umma_sdesc_sw128(v_s + kk * 16 * 128, Gm::KCH, 1024);
                    umma_f16_ts(d, a_t + kk * 8, vb, idO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (j == nktx[x] - 1) umma_commit(&tb[3 * x + 2]);
                if (x == 1 || j >= nkb) umma_commit(&v_empty[j % R]);  // last reader of V(j)
            };
            // operands ready: landed (16-bit cache) or turned into f16 (code cache)
            uint64_t* q_ready = FP8 ? q_conv : q_full;
            uint64_t* k_ready = FP8 ? k_conv : k_full;
            uint64_t* v_ready = FP8 ? v_conv : v_full;
            bool ok = mbar_wait_ns(q_ready, 0, WAIT_NS) && mbar_wait_ns(&k_ready[0], 0, WAIT_NS);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                if (nkb > 0) issue_s(1, 0);
            }
            for (int k = 0; ok && k < nka; ++k) {
                ok = !*abort_flag && mbar_wait_ns(&tb[1], (uint32_t)k & 1u, WAIT_NS) &&
                     mbar_wait_ns(&v_ready[k % R], (uint32_t)(k / R) & 1u, WAIT_NS);
                if (!ok) break;
                tc_fence_after();
                issue_pv(0, k);
                const bool more = k + 1 < nka;
                if (more) {
                    ok = mbar_wait_ns(&k_ready[(k + 1) % R], (uint32_t)((k + 1) / R) & 1u, WAIT_NS);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(0, k + 1);
                }
                if (k < nkb) {
                    ok = mbar_wait_ns(&tb[4], (uint32_t)k & 1u, WAIT_NS);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(1, k);
                    if (k + 1 < nkb) issue_s(1, k + 1);
                }
            }
            if (!ok) fail();
        }
    } else {
        // ---------------- softmax + epilogue of tile X: one query row per thread
        const int x = warp >> 2;
        const int wq = warp & 3;  // tensor-memory lane quarter of this warp
        const int my_nkt = nktx[x];
        uint64_t* s_full = &tb[3 * x];
        uint64_t* p_full = &tb[3 * x + 1];
        uint64_t* o_done = &tb[3 * x + 2];
        const int m = threadIdx.x - 128 * x;
        const bool valid = x < ntiles && m < tnx[x] * G;
        const int ti = valid ? m / G : 0, gh = valid ? m - (m / G) * G : 0;
        const int prow = p.causal ? psx[x] + ti : L - 1;
        const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16) + 256u * x;
        const float sl = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        if constexpr (FP8) {
            // the MMAs run in f16 over a code cache: bf16 queries are turned
            // into f16 in place (both Q tiles, 16-byte pieces over the 256
            // softmax threads); f16 queries are used as they land
            if (!mbar_wait_ns(q_full, 0, WAIT_NS)) {
                ok = false;
            } else if (std::is_same<T, __nv_bfloat16>::value) {
                for (int e = threadIdx.x; e < 2 * Gm::QT / 16; e += 256) {
                    uint4* pc = reinterpret_cast<uint4*>(base + Gm::Q_OFF) + e;
                    uint4 v = *pc;
                    uint32_t* w = &v.x;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float lo = __uint_as_float(w[t] << 16), hi = __uint_as_float(w[t] & 0xffff0000u);
                        w[t] = pack2<__half>(lo, hi);
                    }
                    *pc = v;
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(q_conv);
        }
        for (int kt = 0; kt < my_nkt; ++kt) {
            // S_X(kt) complete; its commit also covers P V_X(kt-1), so O and
            // the P columns are free once this wait returns
            if (*abort_flag || !mbar_wait_ns(s_full, (uint32_t)kt & 1u, WAIT_NS)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kbase = kt * BK;
            // Mask only on tiles that reach past the row's last visible key
            // (the causal diagonal or the context end): `vis` = the last
            // visible column of this tile.  Rows that hold no query of this
            // request are never stored; they take the unmasked path with
            // their warp instead of splitting it.
            const int vis = valid ? min(prow - kbase, BK - 1) : BK - 1;
            const bool full = vis == BK - 1;  // no masked column (most tiles)
            // Exponentials are taken against the row's running maximum
            // m_used (exp2 domain), which a row keeps until a tile's maximum
            // exceeds it by more than 8 (P then stays below 2^8, far inside
            // its type's range).  So once every row of the warp has a
            // maximum, one pass over the scores gives the exponentials and
            // their sum, which bounds them; only the first tile, a tile whose
            // sum says it may outgrow some row's maximum, or a non-positive
            // scale takes the maximum and then the exponentials.  Whether to
            // redo is decided per warp (tensor-memory loads are warp-wide); a
            // row whose maximum did not grow recomputes the same values.
            // 64 scores per tensor-memory wait; P (two per column) is kept in
            // registers until it is final, then written over the low half of
            // the S columns; masked keys get exactly 0.
            float sum = 0.f;
            float pk[BK / 2];  // the tile's P, two per 32-bit column, stored once it is final
            auto exp_pass = [&](float neg_m) {
                sum = 0.f;
#pragma unroll
                for (int q64 = 0; q64 < BK / 64; ++q64) {
                    float a[64];
                    tmem_ld32(t_lane + S_COL + 64 * q64, *reinterpret_cast<float(*)[32]>(a));
                    tmem_ld32(t_lane + S_COL + 64 * q64 + 32, *reinterpret_cast<float(*)[32]>(a + 32));
                    tmem_wait_ld();
                    if (full) {
                        // two scores per fma and two exponents per add (packed fp32x2)
                        const unsigned long long slv = f32x2_pack(sl, sl), nmv = f32x2_pack(neg_m, neg_m);
                        unsigned long long s2 = f32x2_pack(0.f, 0.f);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            float x0, x1;
                            f32x2_unpack(fma_f32x2(f32x2_pack(a[2 * j], a[2 * j + 1]), slv, nmv), x0, x1);
                            const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
                            s2 = add_f32x2(s2, f32x2_pack(e0, e1));
                            pk[32 * q64 + j] = __uint_as_float(pack2<PT>(e0, e1));
                        }
                        float s0, s1;
                        f32x2_unpack(s2, s0, s1);
                        sum += s0 + s1;
                    } else {
                        const int nv = vis - 64 * q64;  // columns j <= nv are visible
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const bool v0 = 2 * j <= nv, v1 = 2 * j + 1 <= nv;
                            const float e0 = v0 ? fast_exp2(fmaf(a[2 * j], sl, neg_m)) : 0.f;
                            const float e1 = v1 ? fast_exp2(fmaf(a[2 * j + 1], sl, neg_m)) : 0.f;
                            sum += e0 + e1;
                            pk[32 * q64 + j] = __uint_as_float(pack2<PT>(e0, e1));
                        }
                    }
                }
            };
            // the maximum alone (first tile; non-positive scale)
            auto max_pass = [&]() -> float {
                float m_t = -INFINITY;
#pragma unroll
                for (int q64 = 0; q64 < BK / 64; ++q64) {
                    float a[64];
                    tmem_ld32(t_lane + S_COL + 64 * q64, *reinterpret_cast<float(*)[32]>(a));
                    tmem_ld32(t_lane + S_COL + 64 * q64 + 32, *reinterpret_cast<float(*)[32]>(a + 32));
                    tmem_wait_ld();
                    const int nv = full ? BK : vis - 64 * q64;
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        if (j <= nv) m_t = fmaxf(m_t, sl > 0.f ? a[j] : a[j] * sl);
                }
                return sl > 0.f ? m_t * sl : m_t;
            };
            // a positive scale keeps the order, so the maximum is taken on raw scores
            const bool have_max = sl > 0.f && __all_sync(0xffffffffu, m_used != -INFINITY);
            float m_tile = have_max ? -INFINITY : max_pass();
            bool grow = false, settled = !have_max;  // settled: this tile's exponent base is final
            float alpha = 1.f;
            auto settle = [&]() {
                const float m_new = fmaxf(m_used, m_tile);
                grow = (m_used == -INFINITY) || (m_new > m_used + 8.f);
                if (grow) {
                    alpha = fast_exp2(m_used - m_new);
                    m_used = m_new;
                }
            };
            if (settled) settle();
            // One call site of the pass.  A row's exponents sum to at least
            // their maximum, so a sum of at most 2^8 proves that no score of
            // the tile exceeded the row's maximum by more than 8: the pass
            // stands.  Otherwise (rare: the tile outgrew some row's maximum,
            // or many scores sit just above it) the tile's maximum is taken
            // and the pass redone against it.
#pragma unroll 1
            for (;;) {
                exp_pass(-m_used);
                if (settled || __all_sync(0xffffffffu, !(sum > 256.f))) break;
                m_tile = max_pass();
                settled = true;
                settle();
            }
            // P over the first 64 S columns, all of which have been read
            tmem_st32(t_lane + P_COL, *reinterpret_cast<float(*)[32]>(pk));
            tmem_st32(t_lane + P_COL + 32, *reinterpret_cast<float(*)[32]>(pk + 32));
            l = l * alpha + sum;
            const bool rescale = __any_sync(0xffffffffu, grow && kt > 0);
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
            }
            tmem_wait_st();
            // Keys at or past L hold no context: their V rows of the tile that
            // holds the context end are zeroed once, by tile A's warps (tile A
            // reads every key tile tile B reads); tile B waits for that.
            if (!FP8 && kt == klast && L - kbase < BK) {  // (a code cache's converter zeroes them)
                if (x == 0) {
                    if (!mbar_wait_ns(&v_full[kt % R], (uint32_t)(kt / R) & 1u, WAIT_NS)) {
                        ok = false;
                        break;
                    }
                    const int keep = L - kbase;
                    uint8_t* v_t = base + Gm::V_OFF + (kt % R) * Gm::TILE;
                    const int rows = BK - keep;
                    for (int e = m; e < rows * Gm::CH * 8; e += 128) {
                        const int c = e / (rows * 8), rem = e - c * rows * 8, r = keep + rem / 8, q16 = rem & 7;
                        *reinterpret_cast<uint4*>(v_t + c * Gm::KCH + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(v_zeroed);
                } else if (!mbar_wait_ns(v_zeroed, 0, WAIT_NS)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (my_nkt > 0) {
            if (ok && !*abort_flag && mbar_wait_ns(o_done, 0, WAIT_NS)) {
                tc_fence_after();
                const float inv = 1.f / l;
                T* orow = static_cast<T*>(p.out) +
                          ((int64_t)(qrx[x] + ti) * p.num_heads + (int64_t)kvh * G + gh) * HD;
#pragma unroll 1
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
            } else {
                fail();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

// The work plan (one CTA): every prefill tile pair of the batch, sorted by
// the number of 128-key tiles its tile A reads, most first (a counting sort
// over kMaxPlanBuckets buckets; the order inside a bucket is whatever the
// atomics give, which changes no output), then the decode rows.  plan[0] =
// pairs, plan[1] = decode rows.
__global__ void __launch_bounds__(1024) varlen_plan_kernel(const int32_t* __restrict__ cu,
                                                           const int32_t* __restrict__ seq_lens, int S, int TT,
                                                           int PW, int causal, int dec_route, int nbuckets,
                                                           int32_t* plan, int4* items, int32_t* dec_req) {
    extern __shared__ int32_t hist[];  // [nbuckets] counts, then [nbuckets] cursors
    __shared__ int32_t n_dec_s;
    int32_t* cursor = hist + nbuckets;
    pdl_wait_primary();
    pdl_launch_dependents();  // the varlen kernel may be scheduled; it waits for this grid
    for (int b = threadIdx.x; b < nbuckets; b += blockDim.x) hist[b] = 0;
    if (threadIdx.x == 0) n_dec_s = 0;
    __syncthreads();
    // 128-key tiles tile A of pair pr of a request reads
    auto tiles_of = [&](int n, int L, int pr) -> int {
        const int ntile = (n + TT - 1) / TT, ta = ntile - 1 - PW * pr, t0 = ta * TT;
        const int kv_end = causal ? L - n + t0 + min(TT, n - t0) : L;
        return min((kv_end + BK - 1) / BK, nbuckets - 1);
    };
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        const int n = cu[i + 1] - cu[i], L = seq_lens[i];
        if (dec_route && n == 1) {
            dec_req[atomicAdd(&n_dec_s, 1)] = i;
            continue;
        }
        const int npair = (n + PW * TT - 1) / (PW * TT);
        for (int pr = 0; pr < npair; ++pr) atomicAdd(&hist[tiles_of(n, L, pr)], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // exclusive prefix over the buckets, longest first
        const int lane = threadIdx.x, per = (nbuckets + 31) / 32;
        const int lo = lane * per, hi = min(nbuckets, lo + per);
        int sum = 0;
        for (int k = lo; k < hi; ++k) sum += hist[nbuckets - 1 - k];
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - sum;
        for (int k = lo; k < hi; ++k) {
            cursor[nbuckets - 1 - k] = run;
            run += hist[nbuckets - 1 - k];
        }
        if (lane == 31) plan[0] = run;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        const int n = cu[i + 1] - cu[i], L = seq_lens[i];
        if (dec_route && n == 1) continue;
        const int npair = (n + PW * TT - 1) / (PW * TT);
        const int q0 = cu[i], ntile = (n + TT - 1) / TT;
        for (int pr = 0; pr < npair; ++pr) {
            const int t0 = (ntile - 1 - PW * pr) * TT;  // tile A's first new token
            items[atomicAdd(&cursor[tiles_of(n, L, pr)], 1)] =
                make_int4(i, q0 + t0, L - n + t0, L | (PW == 2 && t0 >= TT ? (int)0x80000000u : 0));
        }
    }
    if (threadIdx.x == 0) plan[1] = n_dec_s;
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

// dtype: 1 bf16, 2 f16, 3 E4M3 codes (bytes)
bool um_encode(CUtensorMap* m, const void* base, int dtype, const cuuint64_t dims[3], const cuuint64_t strides[2],
               const cuuint32_t box[3], std::string* err) {
    auto fn = um_encode_fn();
    if (!fn) {
        *err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType ty = dtype == 3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : (dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    CUresult r = fn(m, ty, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
        return false;
    }
    return true;
}

// Workspace layout of a planned launch: plan header, prefill items (one per
// possible tile pair, or tile at head_dim 256: the bound below covers both),
// decode-row requests.
int64_t um_pairs_bound(int64_t total_q, int32_t num_seqs, int TT) { return total_q / TT + num_seqs; }
size_t um_round(size_t b) { return (b + 255) & ~(size_t)255; }
size_t um_plan_bytes(int64_t total_q, int32_t num_seqs, int TT) {
    return 256 + um_round((size_t)um_pairs_bound(total_q, num_seqs, TT) * sizeof(int4)) +
           um_round((size_t)num_seqs * sizeof(int32_t));
}

template <typename T, int HD, bool FP8 = false>
cudaError_t um_launch(const AttnArgs& a, int32_t num_blocks, void* workspace, std::string* err,
                      cudaStream_t stream) {
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
    if (FP8) {
        // codes: one 128-byte row per (token, KV head); one box = 16 (or 8) rows
        cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)a.num_kv_heads, (cuuint64_t)num_blocks * a.block_size};
        cuuint64_t strides[2] = {(cuuint64_t)HD, (cuuint64_t)a.num_kv_heads * HD};
        cuuint32_t box[3] = {(cuuint32_t)HD, 1, (cuuint32_t)(a.block_size == 8 ? 8 : BS)};
        if (!um_encode(&tmK, a.k_cache, 3, dims, strides, box, err) ||
            !um_encode(&tmV, a.v_cache, 3, dims, strides, box, err))
            return cudaErrorInvalidValue;
    } else {
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
    p.q = a.q;
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
    p.plan = nullptr;
    p.items = nullptr;
    p.dec_req = nullptr;
    p.k_scales = a.k_scales;
    p.v_scales = a.v_scales;
    // prefill tile pairs (at most total_q / 2T + one per request; single
    // tiles at head_dim 256), then decode CTAs of DG requests; CTAs past the
    // work the kernel finds return
    constexpr int PW = UGeo<HD>::NQ;
    const int64_t pairs = (int64_t)a.total_q / (PW * TT) + a.num_seqs;
    if (pairs >= (1 << kPairBits)) {
        *err = "too many query rows for one varlen launch";
        return cudaErrorInvalidValue;
    }
    const bool dec_route = G <= kMaxDecodeGroupG && HD <= 128;
    const int64_t dgroups = dec_route ? (a.num_seqs + DG - 1) / DG : 0;
    p.dec_ctas = (int32_t)dgroups;
    const size_t smem = um_smem_bytes<HD>(workspace ? 0 : a.num_seqs);
    cudaError_t e = cudaFuncSetAttribute(varlen_umma_kernel<T, HD, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (workspace) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        p.plan = reinterpret_cast<const int32_t*>(ws);
        p.items = reinterpret_cast<const int4*>(ws + 256);
        const int64_t items_cap = um_pairs_bound(a.total_q, a.num_seqs, TT);  // the workspace's layout
        p.dec_req = reinterpret_cast<const int32_t*>(ws + 256 + um_round((size_t)items_cap * sizeof(int4)));
        const int nbuckets = (int)std::min<int64_t>(kMaxPlanBuckets, (int64_t)(a.max_context + BK - 1) / BK + 2);
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3(1);
        pc.blockDim = dim3(1024);
        pc.dynamicSmemBytes = (size_t)2 * nbuckets * sizeof(int32_t);
        pc.stream = stream;
        pc.attrs = attr;
        pc.numAttrs = 1;
        e = cudaLaunchKernelEx(&pc, varlen_plan_kernel, a.cu_seqlens_q, a.seq_lens, a.num_seqs, TT, PW, a.causal,
                               dec_route ? 1 : 0, nbuckets, const_cast<int32_t*>(p.plan),
                               const_cast<int4*>(p.items), const_cast<int32_t*>(p.dec_req));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = workspace ? dim3((unsigned)((pairs + dgroups) * a.num_kv_heads), 1u)
                            : dim3((unsigned)(pairs + dgroups), (unsigned)a.num_kv_heads);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, varlen_umma_kernel<T, HD, FP8>, tmQ, tmK, tmV, p);
}

}  // namespace

bool varlen_umma_supported(int dtype, int head_dim, int block_size, int group, bool kv_fp8) {
    // head_dim 256: block sizes whose 16-token groups are single boxes (a
    // 64-box tile of 8-token blocks would exceed the lanes that issue boxes)
    const bool hd_ok = kv_fp8 ? head_dim == 128 : (head_dim == 64 || head_dim == 128 || head_dim == 256);
    const bool bs_ok = (block_size == 8 && head_dim <= 128) || (block_size % BS == 0 && block_size <= 256);
    return (dtype == 1 || dtype == 2) && hd_ok && bs_ok && group >= 1 && group <= TM;
}

size_t varlen_umma_workspace(int32_t num_seqs, int64_t total_q, int32_t group) {
    if (num_seqs <= 0 || total_q <= 0 || group < 1 || group > TM) return 0;
    return um_plan_bytes(total_q, num_seqs, TM / group);
}

cudaError_t launch_varlen_umma(const AttnArgs& a, int32_t num_blocks, void* workspace, std::string* err,
                               cudaStream_t stream) {
    if (a.total_q == 0 || a.num_seqs == 0) return cudaSuccess;
    auto one = [&](const AttnArgs& c, void* ws) -> cudaError_t {
        if (a.kv_fp8)  // head_dim 128 only
            return a.dtype == 1 ? um_launch<__nv_bfloat16, 128, true>(c, num_blocks, ws, err, stream)
                                : um_launch<__half, 128, true>(c, num_blocks, ws, err, stream);
        if (a.dtype == 1)
            return a.head_dim == 64    ? um_launch<__nv_bfloat16, 64>(c, num_blocks, ws, err, stream)
                   : a.head_dim == 128 ? um_launch<__nv_bfloat16, 128>(c, num_blocks, ws, err, stream)
                                       : um_launch<__nv_bfloat16, 256>(c, num_blocks, ws, err, stream);
        return a.head_dim == 64    ? um_launch<__half, 64>(c, num_blocks, ws, err, stream)
               : a.head_dim == 128 ? um_launch<__half, 128>(c, num_blocks, ws, err, stream)
                                   : um_launch<__half, 256>(c, num_blocks, ws, err, stream);
    };
    if (workspace) return one(a, workspace);  // planned: any number of requests in one launch
    // unplanned: a launch scans at most kMaxSeqsSmem requests in shared
    // memory; query rows keep their global indices (cu_seqlens_q values), so
    // a larger batch runs as several launches over slices of the
    // per-request arrays
    for (int32_t s0 = 0; s0 < a.num_seqs; s0 += kMaxSeqsSmem) {
        AttnArgs c = a;
        c.num_seqs = a.num_seqs - s0 < kMaxSeqsSmem ? a.num_seqs - s0 : kMaxSeqsSmem;
        c.seq_lens = a.seq_lens + s0;
        c.cu_seqlens_q = a.cu_seqlens_q + s0;
        c.block_tables = a.block_tables + (int64_t)s0 * a.max_blocks;
        cudaError_t e = one(c, nullptr);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
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
