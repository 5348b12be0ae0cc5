// pa_decode_tc.cu -- paged decode attention on the tensor cores (bf16/f16).
//
// What it computes is the num_new = 1 case of the handbook's paged_attention
// ("分页 KV Cache", §分页注意力): for sequence s and query head h with KV
// head kv = h / G (G = Hq / Hkv), out = softmax(scale * q K^T) V over the L
// keys of the sequence, K and V read through its block table.
//
// How, on sm_103a:
//  * Work unit = (sequence, KV head); its keys are cut into 16-token tiles
//    (one pool block when block_size is 16, part of one when it is a larger
//    multiple of 16, two blocks when it is 8).  All units' tiles form one
//    flat list of Hkv * sum(ceil(L/16)) tiles, cut into equal contiguous ranges, one per
//    warp of a persistent grid, so every warp streams the same number of
//    bytes whatever the length mix.  A unit cut between warps leaves partial
//    softmax states (m, l, unnormalised o) in the workspace -- written with
//    no fence, count or wait, so a cut costs the streaming warp almost
//    nothing -- and decode_merge_kernel, launched as this kernel's
//    programmatic dependent, merges them by their log-sum-exp in a fixed
//    order once the grid has completed ("aiqz.cc PagedAttention", §工程实现
//    要点: blocks computed apart and merged by the online-softmax rule).  The
//    cut depends only on the lengths, never on physical block ids, so the
//    merge finds every piece from the lengths alone; the workspace holds
//    nothing but the records and never needs clearing.
//  * Each warp runs its own R-deep ring of shared-memory stages (one or two
//    16-token tiles each).  Several lanes issue, in one instruction, the TMA
//    loads (cp.async.bulk.tensor, 128-byte swizzle) of a stage's K and V
//    boxes -- rows of one KV head, gathered through the block table --
//    completing on the stage's mbarrier; block-table entries for the next
//    64 tiles sit in registers.
//  * The G query heads of the unit are packed as the N side of
//    mma.m16n8k16 (padded to 8 or 16): S^T = K Q^T with the 16 tokens as M,
//    so each K/V byte is read once for the whole group; the fp32 scores get
//    an exp2-domain online softmax; P^T is moved into B-fragment layout with
//    movmatrix and O^T += V^T P^T accumulates in fp32 registers.
//  * Tokens past L in a sequence's last block are masked (scores to -inf,
//    V operand lanes to zero) so whatever the unused slots hold never leaks.
//  * Quantized cache (FP8 E4M3 codes, one fp32 scale per token and KV head,
//    scales laid out [num_blocks, num_kv_heads, block_size]; the handbook-
//    adjacent "KV cache：容量推导、分页与回收" names a quantized cache as a
//    per-token size change): the tiles are 1-byte codes (half the bytes of a
//    16-bit cache) and a 1-D bulk copy brings the tile's 16 K and 16 V scales
//    with them.  Codes convert exactly to f16 (cvt e4m3x2 -> f16x2) and feed
//    the same f16 mma.  A key's scale multiplies its score row after the mma;
//    a value's scale multiplies its softmax weight before P is rounded to the
//    f16 operand (the normaliser sums the unscaled weights).  The query is
//    taken as f16(q * scale * log2 e).  The head_dim order inside each mma
//    k-step (keys) and m-tile (values) is permuted -- consistently on both
//    operands, since a dot product does not depend on its order -- so every
//    lane reads contiguous 16-byte pieces of the staged codes.
//  * Pair step (code cache, head_dim 128; a separate instance the host picks
//    for long contexts): when both tiles of a stage belong to one unit they
//    are worked as one 32-token step -- two independent score chains, one
//    softmax reduction and rescale test, sixteen P V products.
//  * Append mode fuses the generation step: the warp that owns a unit's last
//    block patches the new token's K/V row (prefetched from the inputs) into
//    the staged tile before its MMAs and stores the same row to the pool at
//    slot = table[(L-1) / bs] * bs + (L-1) % bs ("分页 KV Cache", §块表与
//    slot mapping) -- slot translation, write and attention in one launch.
//    With a code cache (head_dim 128) the new rows are quantized in the
//    kernel exactly as the quantizing write does, codes and scale going to
//    the pool and to the staged tile.
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

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_decode_status;

constexpr int BS = 16;  // tokens per tile (one m-tile); a pool block holds 8 or 16k tokens

struct TcParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    int32_t max_blocks;
    const int32_t* context_lens;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t group;
    float scale_log2;
    // split merge: two records of group * (HD + 4) floats per warp (slot 0:
    // the warp's first piece, 1: its last), each head's unnormalised o then
    // its m and l
    float* ws_part;  // [total_warps][2]
    // append mode (k_new != nullptr): each sequence's token at position L-1
    // arrives in k_new / v_new [num_seqs, Hkv, HD]; it is written to the pool
    // and attended from these rows, not from the pool
    const void* k_new;
    const void* v_new;
    void* k_pool;
    void* v_pool;
    int32_t block_size;  // tokens per pool block: 8, or a multiple of 16 up to 256
    // quantized cache only: fp32 scales [num_blocks, num_kv_heads, block_size]
    const float* k_scales;
    const float* v_scales;
};

// Warps per CTA, stages per warp, 16-token tiles per stage, and CTAs per SM
// the register budget is sized for (__launch_bounds__).  A stage of about
// 8 KB keeps the per-stage costs (barrier round trip, copy issue) small
// against the bytes it brings: 16-bit head_dim-128 tiles are 8 KB, code
// tiles half that, so code stages hold two tiles.  16-bit head_dim 128: one
// CTA of 8 warps x 2 stages per SM, 128 KB in flight per SM -- measured
// against 8, 10, 12, 16 and 24 stages per SM with 4-16 warps, this is the
// fastest on the GQA, long-context and MHA batches (88.8 / 175.9 / 192.4 us
// against 94.7 / 188.4 / 207.1 us for 2 CTAs x 4 warps x 3 stages): once HBM
// is saturated, more bytes in flight only lengthen the queues, which shows
// at the start and in the tail.  The code path is bound by its per-tile
// conversion chain rather than by memory, so it runs three CTAs (12 warps)
// per SM on two stages each (measured: 12 warps beat 8 and 16 on the
// 64-sequence GQA batch).
template <int HD, bool FP8> struct Pipe;
template <> struct Pipe<64, false> { static constexpr int NW = 4, R = 6, TPS = 1, MINB = 1; };
template <> struct Pipe<128, false> { static constexpr int NW = 8, R = 2, TPS = 1, MINB = 1; };
template <> struct Pipe<256, false> { static constexpr int NW = 2, R = 3, TPS = 1, MINB = 1; };
template <> struct Pipe<128, true> { static constexpr int NW = 4, R = 2, TPS = 2, MINB = 3; };
template <> struct Pipe<256, true> { static constexpr int NW = 4, R = 3, TPS = 1, MINB = 1; };

template <int HD, bool FP8>
struct Geo {
    static constexpr int ELT = FP8 ? 1 : 2;     // bytes per cached element
    static constexpr int CH = HD * ELT / 128;   // 128-byte chunks in one head's row
    static constexpr int TILE = BS * HD * ELT;  // bytes of a K (or V) tile
    static constexpr int TPS = Pipe<HD, FP8>::TPS;
    static constexpr int STAGE = TPS * 2 * TILE;  // per tile: K tile then V tile
    static constexpr int TSCL = FP8 ? 2 * BS : 0;  // floats per tile: 16 K then 16 V scales
    static constexpr int SCL = TPS * TSCL * 4;     // scale bytes of a stage
    static constexpr int KS = HD / 16;           // k-steps of K Q^T == m-tiles of V^T P^T
};

template <int HD, bool FP8>
constexpr size_t smem_bytes(int num_seqs) {
    return 1024 /* alignment slack */ +
           (size_t)Pipe<HD, FP8>::NW * Pipe<HD, FP8>::R * (Geo<HD, FP8>::STAGE + Geo<HD, FP8>::SCL + 8) +
           (size_t)(num_seqs + 1) * 4 + (size_t)num_seqs * 4;
}



// 16-token tiles per sequence and their exclusive prefix over the batch,
// into shared memory (prefix[S + 1]; lens[S] gets the lengths unless null).
// Every thread of the block calls it; it ends with a block barrier.
__device__ __forceinline__ void tile_prefix(const int32_t* context_lens, int S, int32_t* prefix, int32_t* lens) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int L = context_lens[s];
        if (lens) lens[s] = L;
        prefix[s + 1] = L > 0 ? (L + BS - 1) / BS : 0;
    }
    if (threadIdx.x == 0) prefix[0] = 0;
    __syncthreads();
    if (warp == 0) {
        const int per = (S + 31) / 32;
        const int lo = 1 + lane * per, hi = min(S + 1, lo + per);
        int sum = 0;
        for (int i = lo; i < hi; ++i) sum += prefix[i];
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - sum;
        for (int i = lo; i < hi; ++i) {
            run += prefix[i];
            prefix[i] = run;
        }
    }
    __syncthreads();
}

// 16 bytes global -> shared, asynchronously (L2 only).
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
// Arrive on bar once this thread's earlier cp.async copies have landed (the
// barrier counts the arrival among those it expects).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Block sizes a 16-row (or two 8-row) TMA box per 128-byte chunk can load;
// the others are gathered row by row.
__host__ __device__ constexpr bool tma_block_size(int bs) { return bs == 8 || (bs % 16 == 0 && bs <= 256); }

// T: element type of q and out.  FP8: the cache holds E4M3 codes plus
// scales (the mma then runs in f16 whatever T is).  GATHER (16-bit caches
// whose block size no TMA box fits, e.g. 1, 2, 4 or 24): each stage's tile
// is gathered with 16-byte cp.async copies, one token row at a time
// through the block table, into the same swizzled layout the TMA boxes
// give; the stage's barrier then counts one arrival per lane.
template <typename T, int HD, int NT, bool FP8, bool PAIR, bool GATHER = false>
__global__ void __launch_bounds__(Pipe<HD, FP8>::NW * 32, Pipe<HD, FP8>::MINB)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const TcParams p) {
    static_assert(!(GATHER && FP8), "code caches are loaded by TMA only");
    using Gm = Geo<HD, FP8>;
    constexpr int NW = Pipe<HD, FP8>::NW, R = Pipe<HD, FP8>::R, KS = Gm::KS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* scl = reinterpret_cast<float*>(base + (size_t)NW * R * Gm::STAGE);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + (size_t)NW * R * (Gm::STAGE + Gm::SCL));
    int32_t* prefix = reinterpret_cast<int32_t*>(bars + NW * R);
    int32_t* lens = prefix + p.num_seqs + 1;  // context lengths, read once per CTA

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;

    // With programmatic dependent launch this grid may start while the
    // previous kernel on the stream (e.g. the K/V write) is still running;
    // every input is read after this wait.
    if (!GATHER && threadIdx.x == 0) {  // kernel parameters: no need to wait for them
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    pdl_wait_primary();
    // the split merge (the next launch) may be scheduled now; it waits for
    // this grid to complete before it reads anything
    pdl_launch_dependents();

    tile_prefix(p.context_lens, S, prefix, lens);

    const int64_t W = (int64_t)prefix[S] * Hkv;
    // sequences with no context get a zero row (and nothing to merge)
    for (int s = blockIdx.x; s < S; s += gridDim.x) {
        if (prefix[s + 1] == prefix[s]) {
            T* o = static_cast<T*>(p.out) + (int64_t)s * p.num_heads * HD;
            for (int e = threadIdx.x; e < p.num_heads * HD; e += blockDim.x) o[e] = Elt<T>::from_f(0.f);
        }
    }

    const int64_t TW = (int64_t)gridDim.x * NW;
    const int64_t gw = (int64_t)blockIdx.x * NW + warp;
    const int64_t f0 = gw * W / TW, f1 = (gw + 1) * W / TW;
    const int n = (int)(f1 - f0);
    if (n <= 0) return;  // no block-wide barrier follows

    uint64_t* wbar = bars + warp * R;
    uint8_t* wst = base + (size_t)warp * R * Gm::STAGE;
    float* wscl = scl + (size_t)warp * R * (Gm::SCL / 4);
    if (lane == 0) {
        for (int r = 0; r < R; ++r) mbar_init(&wbar[r], GATHER ? 32 : 1);
        mbar_fence_init();
    }
    __syncwarp();

    // flat position -> (sequence, KV head, logical block)
    auto locate = [&](int64_t f, int& s_out, int& h_out, int& b_out) {
        int lo = 0, hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)prefix[mid] * Hkv <= f) lo = mid;
            else hi = mid - 1;
        }
        const int nb = prefix[lo + 1] - prefix[lo];
        const int64_t rem = f - (int64_t)prefix[lo] * Hkv;
        s_out = lo;
        h_out = (int)(rem / nb);
        b_out = (int)(rem - (int64_t)h_out * nb);
    };
    // pool row of the first token of a tile (and, with 8-token blocks, of its
    // second half; that half is never read past the context)
    const int bsz = p.block_size;
    auto table_entry = [&](int64_t rel, int32_t& row2) -> int32_t {
        row2 = 0;
        if (rel >= n) return 0;
        int s, h, t;
        locate(f0 + rel, s, h, t);
        const int32_t* tb = p.block_tables + (int64_t)s * p.max_blocks;
        if (bsz == 8) {
            const int nb8 = (lens[s] + 7) >> 3;
            const int32_t r1 = tb[2 * t] * 8;
            row2 = 2 * t + 1 < nb8 ? tb[2 * t + 1] * 8 : r1;
            return r1;
        }
        const int tok = t * BS;
        return tb[tok / bsz] * bsz + tok % bsz;
    };

    // ---- producer side: issue cursor, table window, TMA
    const uint64_t pol = l2_policy_evict_first();
    int32_t tbl_cur2 = 0, tbl_next2 = 0, tbl_cur = 0, tbl_next = 0;
    if constexpr (!GATHER) {
        tbl_cur = table_entry(lane, tbl_cur2);
        tbl_next = table_entry(32 + lane, tbl_next2);
    }
    int win = 0, ip = 0;
    int is_, ih, ib;
    locate(f0, is_, ih, ib);
    // advance the issue cursor by one tile
    auto advance = [&]() {
        if (++ib == prefix[is_ + 1] - prefix[is_]) {
            ib = 0;
            if (++ih == Hkv) {
                ih = 0;
                do {
                    ++is_;
                } while (is_ < S && prefix[is_ + 1] == prefix[is_]);
            }
        }
    };
    constexpr int TPS = Gm::TPS;
    static_assert(TPS == 1 || TPS == 2, "a stage holds one or two tiles");
    // Issue one stage: tiles ip .. ip+TPS-1 that exist (ip is a multiple of
    // TPS, so they share one 32-tile table window).
    auto issue_next = [&]() {
        if constexpr (GATHER) {
            // one 16-token tile: lane pieces of 16 bytes, K and V rows of
            // token r of the tile from its block (tokens past the context
            // re-read the last one: masked later, and no table entry past
            // ceil(L / bs) is touched)
            const int us = is_, uh = ih, ub = ib;
            advance();
            const int slot = ip % R;
            const int L_u = lens[us];
            const int32_t* tb = p.block_tables + (int64_t)us * p.max_blocks;
            constexpr int PPR = HD * 2 / 16;  // 16-byte pieces of one head's row
            uint8_t* stage = wst + (size_t)slot * Gm::STAGE;
#pragma unroll
            for (int i = 0; i < BS * PPR / 32; ++i) {
                const int pidx = lane + 32 * i, r = pidx / PPR, col16 = pidx - r * PPR;
                const int tok = min(ub * BS + r, L_u - 1);
                const int64_t prow = (int64_t)__ldg(tb + tok / bsz) * bsz + tok % bsz;
                const int64_t off = ((prow * Hkv + uh) * HD) * 2 + col16 * 16;
                const uint32_t dst =
                    smem_u32(stage + (col16 >> 3) * BS * 128 + r * 128 + (((col16 & 7) ^ (r & 7)) << 4));
                cp_async16(dst, static_cast<const uint8_t*>(p.k_pool) + off);
                cp_async16(dst + Gm::TILE, static_cast<const uint8_t*>(p.v_pool) + off);
            }
            cp_async_arrive(&wbar[slot]);
            ++ip;
            return;
        }
        const int w = ip >> 5;
        if (w != win) {
            tbl_cur = tbl_next;
            tbl_cur2 = tbl_next2;
            tbl_next = table_entry((int64_t)(w + 1) * 32 + lane, tbl_next2);
            win = w;
        }
        const int nt_stage = min(TPS, n - ip);
        const int32_t row0 = __shfl_sync(0xffffffffu, tbl_cur, ip & 31);
        const int32_t row20 = __shfl_sync(0xffffffffu, tbl_cur2, ip & 31);
        const int32_t row1 = TPS > 1 ? __shfl_sync(0xffffffffu, tbl_cur, (ip + 1) & 31) : 0;
        const int32_t row21 = TPS > 1 ? __shfl_sync(0xffffffffu, tbl_cur2, (ip + 1) & 31) : 0;
        const int ih0 = ih;
        advance();
        const int ih1 = ih;
        if (TPS > 1 && nt_stage > 1) advance();
        const int slot = (ip / TPS) % R;
        // The stage's copies go out from several lanes in one instruction
        // (a TMA unit takes lane-parallel copies faster than a sequence of
        // copies from one thread): per tile, nbox lanes each load one
        // 128-byte x 16-row (or 8-row) box of K or V, and (code tiles) the
        // next lanes its K and V scales.
        const int halves = bsz == 8 ? 2 : 1;  // 8-token blocks: two 8-row boxes per chunk
        const int nbox = Gm::CH * 2 * halves;
        const int per = nbox + (FP8 ? 2 * halves : 0);
        if (lane == 0) mbar_arrive_expect_tx(&wbar[slot], nt_stage * (2 * Gm::TILE + Gm::TSCL * 4));
        const int j = lane / per, o = lane - j * per;
        if (j < nt_stage) {
            const int32_t row = j ? row1 : row0, row2 = j ? row21 : row20;
            const int ihj = j ? ih1 : ih0;
            fence_proxy_async_smem();
            if (o < nbox) {
                const int hf = o % halves, c = (o / halves) % Gm::CH, is_v = o / (halves * Gm::CH);
                uint8_t* dst = wst + (size_t)slot * Gm::STAGE + j * 2 * Gm::TILE + is_v * Gm::TILE + c * BS * 128 +
                               hf * 1024;
                tma_load_3d(dst, is_v ? &tmV : &tmK, &wbar[slot], 0, ihj * Gm::CH + c, hf ? row2 : row, pol);
            } else if constexpr (FP8) {
                // scales of pool row r for KV head ihj: [r / bs][ihj][r % bs]
                const int q = o - nbox, hf = q % halves, is_v = q / halves;
                const int32_t r = hf ? row2 : row;
                const int64_t si = (int64_t)(r / bsz) * Hkv * bsz + (int64_t)ihj * bsz + r % bsz;
                float* sd = wscl + slot * (Gm::SCL / 4) + j * Gm::TSCL + is_v * BS + hf * 8;
                bulk_g2s(sd, (is_v ? p.v_scales : p.k_scales) + si, halves == 2 ? 32 : 64, &wbar[slot]);
            }
        }
        ip += nt_stage;
    };
    for (int r = 0; r < R && ip < n; ++r) issue_next();

    // ---- consumer side
    const int g = lane >> 2, c4 = lane & 3;
    // ldmatrix lane roles: matrix mi = lane / 8, row ri = lane % 8
    const int mi = lane >> 3, ri = lane & 7;
    // K (non-transposed A operand): token = (mi & 1) * 8 + ri, dims + (mi >> 1) * 8
    const int k_tok = (mi & 1) * 8 + ri, k_dof = (mi >> 1) * 8;
    // V^T (transposed A operand): token = (mi >> 1) * 8 + ri, dims + (mi & 1) * 8
    const int v_tok = (mi >> 1) * 8 + ri, v_dof = (mi & 1) * 8;
    auto swz = [](int tok, int dstart) -> uint32_t {
        const int c = dstart >> 6, j = (dstart & 63) >> 3;
        return (uint32_t)(c * BS * 128 + tok * 128 + ((j ^ (tok & 7)) << 4));
    };

    float acc[KS][NT][4];
    float mrow[NT][2], lrow[NT][2];
    uint32_t qb[KS][NT][2];
    // append mode: this lane's 16-byte pieces of the new K and V rows of the
    // unit's head (HD / 8 pieces each), and the pool block holding position L-1
    constexpr int PPT = HD / 8;
    constexpr int NPC = (2 * PPT + 31) / 32;
    uint4 newp[NPC];
    int32_t last_phys = 0;

    int cs, ch, cb;
    locate(f0, cs, ch, cb);
    int seg_b0 = cb, Lcur = lens[cs];
    bool first_seg = true;
    const T* qbase = static_cast<const T*>(p.q);

    // Quantized cache: lane (g, c4) takes head dims [c4 HD/4, (c4+1) HD/4) of
    // key rows g and g+8, four per k-step (k-step kk: the mma's k pair
    // 2c4, 2c4+1 holds dims kb0 + 4kk, +1 and the pair 2c4+8, +9 holds
    // dims kb0 + 4kk + 2, +3), and head dims [g HD/8, (g+1) HD/8) of value
    // rows 2c4, 2c4+1, 2c4+8, 2c4+9 (m-tile mt, row g + 8hi: dim vb0 + 2mt + hi).
    const int kb0 = c4 * (HD / 4), vb0 = g * (HD / 8);

    // the new token's K/V rows of unit (cs, ch), and the pool block of position L-1
    auto load_new_rows = [&]() {
#pragma unroll
        for (int k = 0; k < NPC; ++k) {
            const int i = lane + 32 * k;
            if (i < 2 * PPT) {
                const uint8_t* src = static_cast<const uint8_t*>(i < PPT ? p.k_new : p.v_new) +
                                     ((int64_t)cs * Hkv + ch) * HD * 2 + (i % PPT) * 16;
                newp[k] = *reinterpret_cast<const uint4*>(src);
            }
        }
        last_phys = p.block_tables[(int64_t)cs * p.max_blocks + (lens[cs] - 1) / bsz];
    };

    auto begin_unit = [&]() {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hh = nt * 8 + g;
                if (hh < G) {
                    const T* qrow = qbase + ((int64_t)cs * p.num_heads + ch * G + hh) * HD;
                    if constexpr (FP8) {
                        float x[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) x[e] = Elt<T>::to_f(qrow[kb0 + 4 * kk + e]) * p.scale_log2;
                        qb[kk][nt][0] = pack2<__half>(x[0], x[1]);
                        qb[kk][nt][1] = pack2<__half>(x[2], x[3]);
                    } else {
                        const T* qp = qrow + kk * 16 + 2 * c4;
                        qb[kk][nt][0] = *reinterpret_cast<const uint32_t*>(qp);
                        qb[kk][nt][1] = *reinterpret_cast<const uint32_t*>(qp + 8);
                    }
                } else {
                    qb[kk][nt][0] = qb[kk][nt][1] = 0u;
                }
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mrow[nt][0] = mrow[nt][1] = -INFINITY;
            lrow[nt][0] = lrow[nt][1] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) acc[kk][nt][0] = acc[kk][nt][1] = acc[kk][nt][2] = acc[kk][nt][3] = 0.f;
        }
        if (p.k_new != nullptr) load_new_rows();
    };

    // head dim of accumulator row g + 8 hi of m-tile mt
    auto odim = [&](int mt, int hi) -> int { return FP8 ? vb0 + 2 * mt + hi : mt * 16 + g + 8 * hi; };

    auto finalize = [&](int bend, int nb) {
        float lt[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = lrow[nt][e];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                lt[nt][e] = l;
            }
        const bool complete = (seg_b0 == 0 && bend == nb);
        if (complete) {
            T* out = static_cast<T*>(p.out) + ((int64_t)cs * p.num_heads + (int64_t)ch * G) * HD;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int hh = nt * 8 + 2 * c4 + e;
                    if (hh < G) {
                        const float inv = 1.f / lt[nt][e];
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            out[hh * HD + odim(mt, 0)] = Elt<T>::from_f(acc[mt][nt][e] * inv);
                            out[hh * HD + odim(mt, 1)] = Elt<T>::from_f(acc[mt][nt][2 + e] * inv);
                        }
                    }
                }
        } else {
            // a piece of a unit cut between warps: its partial state goes to
            // this warp's record (slot 0: the warp's first piece, 1: its
            // last); decode_merge_kernel combines the pieces after this grid
            const int slot = first_seg ? 0 : 1;
            float* rec = p.ws_part + (gw * 2 + slot) * (int64_t)G * (HD + 4);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int hh = nt * 8 + 2 * c4 + e;
                    if (hh < G) {
                        float* r = rec + hh * (HD + 4);
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            r[odim(mt, 0)] = acc[mt][nt][e];
                            r[odim(mt, 1)] = acc[mt][nt][2 + e];
                        }
                        if (g == 0) {
                            r[HD] = mrow[nt][e];
                            r[HD + 1] = lt[nt][e];
                        }
                    }
                }
        }
    };

    begin_unit();
    const uint32_t st0 = smem_u32(wst);
    for (int i = 0; i < n; ++i) {
        const int stg = i / TPS, sub = i - stg * TPS, slot = stg % R;
        if (sub == 0 && !mbar_wait_bounded(&wbar[slot], (uint32_t)(stg / R) & 1u, kMaxPolls)) {
            if (lane == 0) atomicOr(&g_decode_status, kStatusTimeout);
            for (int sj = stg + 1; sj * TPS < ip; ++sj)
                mbar_wait_bounded(&wbar[sj % R], (uint32_t)(sj / R) & 1u, kMaxPolls);
            return;
        }
        const uint32_t kt = st0 + (uint32_t)slot * Gm::STAGE + sub * 2 * Gm::TILE, vt = kt + Gm::TILE;
        const int valid = min(BS, Lcur - cb * BS);
        if (!FP8 && p.k_new != nullptr && cb == prefix[cs + 1] - prefix[cs] - 1) {
            // the new token: into the staged tiles (its attention input) and the pool
            const int r = valid - 1;
            const int64_t slot_row = (int64_t)last_phys * bsz + (Lcur - 1) % bsz;
#pragma unroll
            for (int k = 0; k < NPC; ++k) {
                const int i = lane + 32 * k;
                if (i < 2 * PPT) {
                    const int j = i % PPT, c = j >> 3, q16 = j & 7;
                    const uint32_t dst = (i < PPT ? kt : vt) + c * BS * 128 + r * 128 + ((q16 ^ (r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(newp[k].x),
                                 "r"(newp[k].y), "r"(newp[k].z), "r"(newp[k].w)
                                 : "memory");
                    uint8_t* pool = static_cast<uint8_t*>(i < PPT ? p.k_pool : p.v_pool);
                    *reinterpret_cast<uint4*>(pool + (slot_row * Hkv + ch) * HD * 2 + j * 16) = newp[k];
                }
            }
            __syncwarp();
        }
        if constexpr (FP8 && HD == 128) {
            if (p.k_new != nullptr && cb == prefix[cs + 1] - prefix[cs] - 1) {
                // the new token, quantized as the quantizing write does it
                // (scale = max|x| / 448, code = E4M3(x / scale)): lanes 0-15
                // hold 8 elements each of the K row, lanes 16-31 of the V
                // row; codes and scale go to the pool and the staged tile.
                static_assert(NPC == 1 && PPT == 16, "one 16-byte piece of the new rows per lane");
                const int r = valid - 1, j = lane & 15, is_v = lane >> 4;
                const int64_t off = (Lcur - 1) % bsz, slot_row = (int64_t)last_phys * bsz + off;
                float x[8], amax = 0.f;
                const uint32_t w4[4] = {newp[0].x, newp[0].y, newp[0].z, newp[0].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const T lo = *reinterpret_cast<const T*>(&w4[e]);
                    const T hi = *(reinterpret_cast<const T*>(&w4[e]) + 1);
                    x[2 * e] = Elt<T>::to_f(lo);
                    x[2 * e + 1] = Elt<T>::to_f(hi);
                    amax = fmaxf(amax, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
                }
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const float sq = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
                uint32_t cw[2] = {0u, 0u};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    cw[e >> 2] |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[e], sq), __NV_SATFINITE, __NV_E4M3)
                                  << (8 * (e & 3));
                uint8_t* pool = static_cast<uint8_t*>(is_v ? p.v_pool : p.k_pool);
                *reinterpret_cast<uint2*>(pool + (slot_row * Hkv + ch) * HD + 8 * j) = make_uint2(cw[0], cw[1]);
                const int b = 8 * j;
                const uint32_t dst = (is_v ? vt : kt) + r * 128 + ((((b & 127) >> 4) ^ (r & 7)) << 4) + (b & 15);
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(dst), "r"(cw[0]), "r"(cw[1]) : "memory");
                if (j == 0) {
                    float* sp = const_cast<float*>(is_v ? p.v_scales : p.k_scales);
                    sp[((int64_t)last_phys * Hkv + ch) * bsz + off] = sq;
                    wscl[slot * (Gm::SCL / 4) + sub * Gm::TSCL + is_v * BS + r] = sq;
                }
                __syncwarp();
            }
        }

        if constexpr (FP8 && TPS == 2 && PAIR) {
            // Pair step: when both tiles of this stage belong to the unit (and
            // the second is not the one the new token goes to), they are
            // worked as one 32-token step: two independent score chains, one
            // softmax reduction and rescale, then sixteen P V products.  Tile
            // a (this one) is full; tile b may end the context.
            const int nb_u = prefix[cs + 1] - prefix[cs];
            if (sub == 0 && i + 1 < n && cb + 1 < nb_u && !(p.k_new != nullptr && cb + 1 == nb_u - 1)) {
                const uint32_t ktb = kt + 2 * Gm::TILE, vtb = ktb + Gm::TILE;
                const int valid_b = min(BS, Lcur - (cb + 1) * BS);
                float sa[NT][4], sb[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
                constexpr int KP = HD / 64;
#pragma unroll
                for (int u = 0; u < KP; ++u) {
                    uint4 wa[2], wb[2];
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        const int r = g + 8 * hi, b = kb0 + 16 * u;
                        const uint32_t off = (b >> 7) * BS * 128 + r * 128 + ((((b & 127) >> 4) ^ (r & 7)) << 4);
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(wa[hi].x), "=r"(wa[hi].y), "=r"(wa[hi].z), "=r"(wa[hi].w) : "r"(kt + off));
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(wb[hi].x), "=r"(wb[hi].y), "=r"(wb[hi].z), "=r"(wb[hi].w) : "r"(ktb + off));
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int kk = 4 * u + q4;
                        const uint32_t a0w = (&wa[0].x)[q4], a1w = (&wa[1].x)[q4];
                        const uint32_t b0w = (&wb[0].x)[q4], b1w = (&wb[1].x)[q4];
                        uint32_t a0, a2;
                        e4m3x4_to_f16x2x2(a0w, a0, a2);
                        uint32_t a1, a3;
                        e4m3x4_to_f16x2x2(a1w, a1, a3);
                        uint32_t b0, b2;
                        e4m3x4_to_f16x2x2(b0w, b0, b2);
                        uint32_t b1, b3;
                        e4m3x4_to_f16x2x2(b1w, b1, b3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma16816<__half>(sa[nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
                            mma16816<__half>(sb[nt], b0, b1, b2, b3, qb[kk][nt][0], qb[kk][nt][1]);
                        }
                    }
                }
                const float* ssa = wscl + slot * (Gm::SCL / 4);  // tile a's K then V scales
                const float* ssb = ssa + Gm::TSCL;                // tile b's
                const bool okb0 = g < valid_b, okb1 = g + 8 < valid_b;
                const float ka0 = ssa[g], ka1 = ssa[g + 8], kb0s = ssb[g], kb1s = ssb[g + 8];
                const float va0 = ssa[BS + g], va1 = ssa[BS + g + 8];
                const float vb0s = okb0 ? ssb[BS + g] : 0.f, vb1s = okb1 ? ssb[BS + g + 8] : 0.f;
                uint32_t pa[NT][2], pbb[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float xa0 = sa[nt][0] * ka0, xa1 = sa[nt][1] * ka0, xa2 = sa[nt][2] * ka1, xa3 = sa[nt][3] * ka1;
                    const float xb0 = okb0 ? sb[nt][0] * kb0s : -INFINITY, xb1 = okb0 ? sb[nt][1] * kb0s : -INFINITY;
                    const float xb2 = okb1 ? sb[nt][2] * kb1s : -INFINITY, xb3 = okb1 ? sb[nt][3] * kb1s : -INFINITY;
                    float mx0 = fmaxf(fmaxf(xa0, xa2), fmaxf(xb0, xb2)), mx1 = fmaxf(fmaxf(xa1, xa3), fmaxf(xb1, xb3));
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(mrow[nt][0], mx0), mn1 = fmaxf(mrow[nt][1], mx1);
                    const float al0 = fast_exp2(mrow[nt][0] - mn0), al1 = fast_exp2(mrow[nt][1] - mn1);
                    mrow[nt][0] = mn0;
                    mrow[nt][1] = mn1;
                    const float pa0 = fast_exp2(xa0 - mn0), pa1 = fast_exp2(xa1 - mn1);
                    const float pa2 = fast_exp2(xa2 - mn0), pa3 = fast_exp2(xa3 - mn1);
                    const float pb0 = fast_exp2(xb0 - mn0), pb1 = fast_exp2(xb1 - mn1);
                    const float pb2 = fast_exp2(xb2 - mn0), pb3 = fast_exp2(xb3 - mn1);
                    lrow[nt][0] = fmaf(lrow[nt][0], al0, (pa0 + pa2) + (pb0 + pb2));
                    lrow[nt][1] = fmaf(lrow[nt][1], al1, (pa1 + pa3) + (pb1 + pb3));
                    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            acc[mt][nt][0] *= al0;
                            acc[mt][nt][1] *= al1;
                            acc[mt][nt][2] *= al0;
                            acc[mt][nt][3] *= al1;
                        }
                    }
                    pa[nt][0] = movm_t(pack2<__half>(pa0 * va0, pa1 * va0));
                    pa[nt][1] = movm_t(pack2<__half>(pa2 * va1, pa3 * va1));
                    pbb[nt][0] = movm_t(pack2<__half>(pb0 * vb0s, pb1 * vb0s));
                    pbb[nt][1] = movm_t(pack2<__half>(pb2 * vb1s, pb3 * vb1s));
                }
                uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
                if (valid_b < BS) {
                    m01 = (2 * c4 < valid_b ? 0x0000ffffu : 0u) | (2 * c4 + 1 < valid_b ? 0xffff0000u : 0u);
                    m23 = (2 * c4 + 8 < valid_b ? 0x0000ffffu : 0u) | (2 * c4 + 9 < valid_b ? 0xffff0000u : 0u);
                }
                constexpr int VP = HD / 128;
#pragma unroll
                for (int u = 0; u < VP; ++u) {
                    uint4 va[4], vb[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int r = 2 * c4 + (t & 1) + 8 * (t >> 1), b = vb0 + 16 * u;
                        const uint32_t off = (b >> 7) * BS * 128 + r * 128 + ((((b & 127) >> 4) ^ (r & 7)) << 4);
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(va[t].x), "=r"(va[t].y), "=r"(va[t].z), "=r"(va[t].w) : "r"(vt + off));
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(vb[t].x), "=r"(vb[t].y), "=r"(vb[t].z), "=r"(vb[t].w) : "r"(vtb + off));
                    }
#pragma unroll
                    for (int mq = 0; mq < 8; ++mq) {
                        const int mt = 8 * u + mq, wi = mq >> 1;
                        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                        const uint32_t la = __byte_perm((&va[0].x)[wi], (&va[1].x)[wi], sel);
                        const uint32_t ha = __byte_perm((&va[2].x)[wi], (&va[3].x)[wi], sel);
                        const uint32_t lb = __byte_perm((&vb[0].x)[wi], (&vb[1].x)[wi], sel);
                        const uint32_t hb = __byte_perm((&vb[2].x)[wi], (&vb[3].x)[wi], sel);
                        uint32_t a0, a1;
                        e4m3x4_to_f16x2x2(la, a0, a1);
                        uint32_t a2, a3;
                        e4m3x4_to_f16x2x2(ha, a2, a3);
                        uint32_t b0, b1;
                        e4m3x4_to_f16x2x2(lb, b0, b1);
                        uint32_t b2, b3;
                        e4m3x4_to_f16x2x2(hb, b2, b3);
                        if (valid_b < BS) {
                            b0 &= m01;
                            b1 &= m01;
                            b2 &= m23;
                            b3 &= m23;
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma16816<__half>(acc[mt][nt], a0, a1, a2, a3, pa[nt][0], pa[nt][1]);
                            mma16816<__half>(acc[mt][nt], b0, b1, b2, b3, pbb[nt][0], pbb[nt][1]);
                        }
                    }
                }
                __syncwarp();
                if (ip < n) issue_next();
                ++i;  // tile b is done too
                cb += 2;
                const bool unit_done = (cb == nb_u);
                if (unit_done || i == n - 1) {
                    finalize(cb, nb_u);
                    first_seg = false;
                    if (unit_done && i < n - 1) {
                        cb = 0;
                        seg_b0 = 0;
                        if (++ch == Hkv) {
                            ch = 0;
                            do {
                                ++cs;
                            } while (cs < S && prefix[cs + 1] == prefix[cs]);
                            Lcur = lens[cs];
                        }
                        begin_unit();
                    }
                }
                continue;
            }
        }

        // S^T = K Q^T : 16 tokens x (8 NT) heads, fp32
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        if constexpr (FP8) {
            constexpr int KP = HD / 64;  // 16-byte pieces of a lane's key bytes per row
            uint4 kw[2][KP];
#pragma unroll
            for (int hi = 0; hi < 2; ++hi)
#pragma unroll
                for (int u = 0; u < KP; ++u) {
                    const int r = g + 8 * hi, b = kb0 + 16 * u;
                    const uint32_t a = kt + (b >> 7) * BS * 128 + r * 128 + ((((b & 127) >> 4) ^ (r & 7)) << 4);
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(kw[hi][u].x), "=r"(kw[hi][u].y), "=r"(kw[hi][u].z), "=r"(kw[hi][u].w)
                                 : "r"(a));
                }
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const uint32_t w0 = (&kw[0][kk >> 2].x)[kk & 3], w1 = (&kw[1][kk >> 2].x)[kk & 3];
                uint32_t a0, a2;
                e4m3x4_to_f16x2x2(w0, a0, a2);
                uint32_t a1, a3;
                e4m3x4_to_f16x2x2(w1, a1, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma16816<__half>(sc[nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kt + swz(k_tok, kk * 16 + k_dof), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816<T>(sc[nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
            }
        }

        // online softmax over this block (exp2 domain)
        const bool ok0 = g < valid, ok1 = g + 8 < valid;
        // score multipliers of rows g, g+8 and (quantized cache) value scales
        float sm0 = p.scale_log2, sm1 = p.scale_log2, vs0 = 1.f, vs1 = 1.f;
        if constexpr (FP8) {
            const float* ss = wscl + slot * (Gm::SCL / 4) + sub * Gm::TSCL;
            sm0 = ss[g];
            sm1 = ss[g + 8];
            vs0 = ok0 ? ss[BS + g] : 0.f;  // a slot past the context may hold anything
            vs1 = ok1 ? ss[BS + g + 8] : 0.f;
        }
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float x0 = ok0 ? sc[nt][0] * sm0 : -INFINITY;
            const float x1 = ok0 ? sc[nt][1] * sm0 : -INFINITY;
            const float x2 = ok1 ? sc[nt][2] * sm1 : -INFINITY;
            const float x3 = ok1 ? sc[nt][3] * sm1 : -INFINITY;
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
            // rescale O only when some row's maximum grew (after the first
            // few tiles it rarely does; the vote is warp-uniform)
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    acc[mt][nt][0] *= al0;
                    acc[mt][nt][1] *= al1;
                    acc[mt][nt][2] *= al0;
                    acc[mt][nt][3] *= al1;
                }
            }
            if constexpr (FP8) {
                pb[nt][0] = movm_t(pack2<__half>(p0 * vs0, p1 * vs0));
                pb[nt][1] = movm_t(pack2<__half>(p2 * vs1, p3 * vs1));
            } else {
                pb[nt][0] = movm_t(pack2<T>(p0, p1));
                pb[nt][1] = movm_t(pack2<T>(p2, p3));
            }
        }

        // O^T += V^T P^T
        uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
        if (valid < BS) {
            m01 = (2 * c4 < valid ? 0x0000ffffu : 0u) | (2 * c4 + 1 < valid ? 0xffff0000u : 0u);
            m23 = (2 * c4 + 8 < valid ? 0x0000ffffu : 0u) | (2 * c4 + 9 < valid ? 0xffff0000u : 0u);
        }
        if constexpr (FP8) {
            constexpr int VP = HD / 128;  // 16-byte pieces of a lane's value bytes per row
            uint4 vw[4][VP];              // rows 2c4, 2c4+1, 2c4+8, 2c4+9
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int u = 0; u < VP; ++u) {
                    const int r = 2 * c4 + (t & 1) + 8 * (t >> 1), b = vb0 + 16 * u;
                    const uint32_t a = vt + (b >> 7) * BS * 128 + r * 128 + ((((b & 127) >> 4) ^ (r & 7)) << 4);
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(vw[t][u].x), "=r"(vw[t][u].y), "=r"(vw[t][u].z), "=r"(vw[t][u].w)
                                 : "r"(a));
                }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                // dims vb0 + 2mt (row g) and + 1 (row g+8): bytes 2mt, 2mt+1 of the lane's value bytes,
                // interleaved token pair by token pair
                const int wi = (2 * mt) >> 2;
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                const uint32_t w0 = (&vw[0][wi >> 2].x)[wi & 3], w1 = (&vw[1][wi >> 2].x)[wi & 3];
                const uint32_t w8 = (&vw[2][wi >> 2].x)[wi & 3], w9 = (&vw[3][wi >> 2].x)[wi & 3];
                const uint32_t lo = __byte_perm(w0, w1, sel), hi = __byte_perm(w8, w9, sel);
                uint32_t a0, a1;
                e4m3x4_to_f16x2x2(lo, a0, a1);
                uint32_t a2, a3;
                e4m3x4_to_f16x2x2(hi, a2, a3);
                if (valid < BS) {
                    a0 &= m01;
                    a1 &= m01;
                    a2 &= m23;
                    a3 &= m23;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma16816<__half>(acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            }
        } else {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vt + swz(v_tok, mt * 16 + v_dof), a0, a1, a2, a3);
                if (valid < BS) {
                    a0 &= m01;
                    a1 &= m01;
                    a2 &= m23;
                    a3 &= m23;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816<T>(acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            }
        }
        __syncwarp();
        if ((sub == TPS - 1 || i == n - 1) && ip < n) issue_next();

        const int nb = prefix[cs + 1] - prefix[cs];
        ++cb;
        const bool unit_done = (cb == nb);
        if (unit_done || i == n - 1) {
            finalize(cb, nb);
            first_seg = false;
            if (unit_done && i < n - 1) {
                cb = 0;
                seg_b0 = 0;
                if (++ch == Hkv) {
                    ch = 0;
                    do {
                        ++cs;
                    } while (cs < S && prefix[cs + 1] == prefix[cs]);
                    Lcur = lens[cs];
                }
                begin_unit();
            }
        }
    }
}

// The split merge ("aiqz.cc PagedAttention", §工程实现要点: blocks computed
// apart, merged by the online-softmax rule).  Launched right after
// decode_tc_kernel as its programmatic dependent; half a warp per (sequence,
// KV head, query head of the group).  Before it waits for the decode grid it
// finds its unit's pieces from the lengths alone, with the decode's own cut
// (warp w owns flat tiles [w W / TW, (w+1) W / TW)): the unit's first warp
// holds it as its first piece (record slot 0) when the unit starts where
// that warp's range starts, else as its last (slot 1); every later warp
// holds it as its first piece.  A unit inside one warp's range was written
// whole by that warp and is skipped.  The lengths were complete before the
// decode grid started (it waited for them), so reading them early is safe.
// After the wait the records are read in batches of up to B whose loads all
// go out together (one memory round trip per batch), each batch folded into
// the running state by the log-sum-exp rule, in warp order.  Warps with
// empty ranges (only when the batch has fewer tiles than the decode grid
// has warps) hold no record.
template <typename T, int HD>
__global__ void __launch_bounds__(256) decode_merge_kernel(const TcParams p, const int64_t TW) {
    constexpr int E = HD / 16;             // output elements per lane
    constexpr int B = HD <= 128 ? 8 : 4;   // records per batch
    extern __shared__ int32_t mprefix[];   // [num_seqs + 1]
    const int S = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
    tile_prefix(p.context_lens, S, mprefix, nullptr);
    const int64_t item = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);
    if (item >= (int64_t)S * Hkv * G) return;
    const int hl = threadIdx.x & 15;  // lane within the half warp
    const int j = (int)(item % G);
    const int64_t u = item / G;
    const int s = (int)(u / Hkv), h = (int)(u - (int64_t)s * Hkv);
    const int nb = mprefix[s + 1] - mprefix[s];
    if (nb == 0) return;  // no context: the decode wrote the zero row
    const int64_t W = (int64_t)mprefix[S] * Hkv;
    const int64_t u0 = (int64_t)mprefix[s] * Hkv + (int64_t)h * nb, u1 = u0 + nb;
    // the warp owning flat tile f: the last w with w W / TW <= f
    auto owner = [&](int64_t f) -> int64_t { return ((f + 1) * TW + W - 1) / W - 1; };
    const int64_t wf = owner(u0), wl = owner(u1 - 1);
    if (wf == wl) return;  // held whole by one warp
    const int slot0 = u0 == wf * W / TW ? 0 : 1;
    const float* rec0 = p.ws_part + (int64_t)j * (HD + 4) + hl * E;
    const int64_t rstride = (int64_t)G * (HD + 4);

    pdl_wait_primary();  // the records are the decode grid's output
    float M = -INFINITY, L = 0.f, o[E];
#pragma unroll
    for (int t = 0; t < E; ++t) o[t] = 0.f;
    for (int64_t w0 = wf; w0 <= wl; w0 += B) {
        float m[B], l[B];
        float4 a[B][E / 4];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int64_t w = w0 + b;
            // an absent record (past the unit, or an empty range) weighs nothing
            const bool ok = w <= wl && !(W < TW && w * W / TW == (w + 1) * W / TW);
            m[b] = -INFINITY;
            l[b] = 0.f;
            if (ok) {
                const float* r = rec0 + (w * 2 + (w == wf ? slot0 : 0)) * rstride;
                m[b] = __ldcg(r - hl * E + HD);
                l[b] = __ldcg(r - hl * E + HD + 1);
#pragma unroll
                for (int t = 0; t < E / 4; ++t) a[b][t] = __ldcg(reinterpret_cast<const float4*>(r) + t);
            } else {
#pragma unroll
                for (int t = 0; t < E / 4; ++t) a[b][t] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float Mn = M;
#pragma unroll
        for (int b = 0; b < B; ++b) Mn = fmaxf(Mn, m[b]);
        const float c = exp2f(M - Mn);
        L *= c;
#pragma unroll
        for (int t = 0; t < E; ++t) o[t] *= c;
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const float e = exp2f(m[b] - Mn);  // 0 for an absent record
            L = fmaf(e, l[b], L);
#pragma unroll
            for (int t = 0; t < E / 4; ++t) {
                o[4 * t + 0] = fmaf(e, a[b][t].x, o[4 * t + 0]);
                o[4 * t + 1] = fmaf(e, a[b][t].y, o[4 * t + 1]);
                o[4 * t + 2] = fmaf(e, a[b][t].z, o[4 * t + 2]);
                o[4 * t + 3] = fmaf(e, a[b][t].w, o[4 * t + 3]);
            }
        }
        M = Mn;
    }
    const float inv = 1.f / L;
    T* out = static_cast<T*>(p.out) + ((int64_t)s * p.num_heads + (int64_t)h * G + j) * HD + hl * E;
#pragma unroll
    for (int t = 0; t < E; t += 4) {  // 4 outputs (8 bytes) per store
        uint2 v;
        v.x = pack2<T>(o[t] * inv, o[t + 1] * inv);
        v.y = pack2<T>(o[t + 2] * inv, o[t + 3] * inv);
        *reinterpret_cast<uint2*>(out + t) = v;
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// The cache as a 3-D tensor: 128 bytes (64 16-bit elements, or 128 E4M3
// codes) x (Hkv * CH) 128-byte chunks of a token row x num_blocks *
// block_size token rows; one box = one chunk of one KV head over the 16 (or
// 8) rows of a block.
bool make_kv_map(CUtensorMap* m, const void* cache, int dtype, bool fp8, int num_blocks, int block_size,
                 int num_kv_heads, int head_dim, std::string* err) {
    auto fn = encode_fn();
    if (!fn) {
        *err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    const int elt = fp8 ? 1 : 2;
    const int ch = head_dim * elt / 128, inner = 128 / elt;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)num_kv_heads * ch, (cuuint64_t)num_blocks * block_size};
    cuuint64_t strides[2] = {128, (cuuint64_t)num_kv_heads * head_dim * elt};
    cuuint32_t box[3] = {(cuuint32_t)inner, 1, (cuuint32_t)(block_size == 8 ? 8 : BS)};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                       : (dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    // L2 fills of 256 bytes suit a 16-bit head row (two 128-byte chunks); a
    // code row is one 128-byte chunk, and a 256-byte fill would drag in the
    // neighbouring head's row
    const CUtensorMapL2promotion promo = fp8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    CUresult r = fn(m, ty, 3, const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
        return false;
    }
    return true;
}

template <typename T, int HD, int NT, bool FP8, bool PAIR = false, bool GATHER = false>
const void* kernel_ptr() {
    return reinterpret_cast<const void*>(&decode_tc_kernel<T, HD, NT, FP8, PAIR, GATHER>);
}

template <int HD, bool FP8>
int grid_for(const void* kfn, int32_t num_seqs, int32_t num_kv_heads, int32_t max_context, int64_t override_ctas) {
    // an explicit grid (PA_OPT_DECODE_CTAS) is capped; each warp owns two split records
    if (override_ctas > 0) return (int)(override_ctas < 16000 ? override_ctas : 16000);
    int dev = 0, sms = 0, occ = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = smem_bytes<HD, FP8>(num_seqs);
    cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kfn, Pipe<HD, FP8>::NW * 32, smem);
    if (occ < 1) occ = 1;
    int64_t grid = (int64_t)sms * occ;
    // at least two blocks per warp on average when every context is max_context long
    const int64_t wmax = (int64_t)num_seqs * num_kv_heads * ((max_context + BS - 1) / BS);
    const int64_t cap = (wmax + 2 * Pipe<HD, FP8>::NW - 1) / (2 * Pipe<HD, FP8>::NW);
    if (grid > cap) grid = cap;
    return (int)(grid < 1 ? 1 : grid);
}

template <typename T, int HD, int NT, bool FP8, bool PAIR = false, bool GATHER = false>
cudaError_t launch_typed(const AttnArgs& a, int32_t num_blocks, int grid, void* workspace, std::string* err,
                         cudaStream_t stream) {
    CUtensorMap tmK, tmV;
    if (GATHER) {  // no boxes: the maps are not read
        memset(&tmK, 0, sizeof(tmK));
        memset(&tmV, 0, sizeof(tmV));
    } else if (!make_kv_map(&tmK, a.k_cache, a.dtype, FP8, num_blocks, a.block_size, a.num_kv_heads, HD, err) ||
               !make_kv_map(&tmV, a.v_cache, a.dtype, FP8, num_blocks, a.block_size, a.num_kv_heads, HD, err)) {
        return cudaErrorInvalidValue;
    }
    TcParams p;
    p.out = a.out;
    p.q = a.q;
    p.block_tables = a.block_tables;
    p.max_blocks = a.max_blocks;
    p.context_lens = a.seq_lens;
    p.num_seqs = a.num_seqs;
    p.num_heads = a.num_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.group = a.num_heads / a.num_kv_heads;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.ws_part = static_cast<float*>(workspace);
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.k_pool = const_cast<void*>(a.k_cache);
    p.v_pool = const_cast<void*>(a.v_cache);
    p.block_size = a.block_size;
    p.k_scales = a.k_scales;
    p.v_scales = a.v_scales;

    const void* kfn = kernel_ptr<T, HD, NT, FP8, PAIR, GATHER>();
    const size_t smem = smem_bytes<HD, FP8>(a.num_seqs);
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the grid may be scheduled while the
    // previous kernel on the stream finishes; the kernel waits for it first
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Pipe<HD, FP8>::NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_tc_kernel<T, HD, NT, FP8, PAIR, GATHER>, tmK, tmV, p);
    if (e != cudaSuccess) return e;
    // the split merge, one warp per (unit, query head), as a programmatic
    // dependent
    const int64_t items = (int64_t)a.num_seqs * a.num_kv_heads * p.group;
    const int64_t tw = (int64_t)grid * Pipe<HD, FP8>::NW;
    cudaLaunchConfig_t mcfg = cfg;
    mcfg.gridDim = dim3((unsigned)((items + 15) / 16));
    mcfg.blockDim = dim3(256);
    mcfg.dynamicSmemBytes = (size_t)(a.num_seqs + 1) * sizeof(int32_t);
    return cudaLaunchKernelEx(&mcfg, decode_merge_kernel<T, HD>, p, tw);
}

template <typename T>
cudaError_t launch_dtype(const AttnArgs& a, int32_t num_blocks, int grid, void* ws, std::string* err,
                         cudaStream_t st) {
    const int G = a.num_heads / a.num_kv_heads;
    const bool two = G > 8;
    if (a.kv_fp8) {
        if (a.head_dim == 128)
            return two ? launch_typed<T, 128, 2, true>(a, num_blocks, grid, ws, err, st)
                       : a.pair_steps ? launch_typed<T, 128, 1, true, true>(a, num_blocks, grid, ws, err, st)
                                      : launch_typed<T, 128, 1, true>(a, num_blocks, grid, ws, err, st);
        return two ? launch_typed<T, 256, 2, true>(a, num_blocks, grid, ws, err, st)
                   : launch_typed<T, 256, 1, true>(a, num_blocks, grid, ws, err, st);
    }
    if (!tma_block_size(a.block_size)) {
        switch (a.head_dim) {
            case 64: return two ? launch_typed<T, 64, 2, false, false, true>(a, num_blocks, grid, ws, err, st)
                                : launch_typed<T, 64, 1, false, false, true>(a, num_blocks, grid, ws, err, st);
            case 128: return two ? launch_typed<T, 128, 2, false, false, true>(a, num_blocks, grid, ws, err, st)
                                 : launch_typed<T, 128, 1, false, false, true>(a, num_blocks, grid, ws, err, st);
            default: return two ? launch_typed<T, 256, 2, false, false, true>(a, num_blocks, grid, ws, err, st)
                                : launch_typed<T, 256, 1, false, false, true>(a, num_blocks, grid, ws, err, st);
        }
    }
    switch (a.head_dim) {
        case 64: return two ? launch_typed<T, 64, 2, false>(a, num_blocks, grid, ws, err, st)
                            : launch_typed<T, 64, 1, false>(a, num_blocks, grid, ws, err, st);
        case 128: return two ? launch_typed<T, 128, 2, false>(a, num_blocks, grid, ws, err, st)
                             : launch_typed<T, 128, 1, false>(a, num_blocks, grid, ws, err, st);
        default: return two ? launch_typed<T, 256, 2, false>(a, num_blocks, grid, ws, err, st)
                            : launch_typed<T, 256, 1, false>(a, num_blocks, grid, ws, err, st);
    }
}

}  // namespace

bool decode_tc_supported(int dtype, int head_dim, int block_size, int group, bool kv_fp8) {
    const bool hd_ok = kv_fp8 ? (head_dim == 128 || head_dim == 256)
                              : (head_dim == 64 || head_dim == 128 || head_dim == 256);
    // 16-bit caches of any block size (boxes or a row gather); code caches by boxes only
    const bool bs_ok = kv_fp8 ? tma_block_size(block_size) : block_size >= 1;
    return (dtype == 1 || dtype == 2) && hd_ok && bs_ok && group >= 1 && group <= 16;
}

int decode_tc_grid(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                   int32_t max_context, int dtype, int32_t group, int64_t ctas_override, bool kv_fp8) {
    const int s = num_seqs < kDecodeMaxSeqsPerLaunch ? num_seqs : kDecodeMaxSeqsPerLaunch;
    const bool two = group > 8;
    const bool bf = dtype == 1;
    if (!kv_fp8 && !tma_block_size(block_size)) {  // the row-gather instances
#define PA_GFN(HD)                                                                                           \
    (bf ? (two ? kernel_ptr<__nv_bfloat16, HD, 2, false, false, true>()                                      \
               : kernel_ptr<__nv_bfloat16, HD, 1, false, false, true>())                                     \
        : (two ? kernel_ptr<__half, HD, 2, false, false, true>() : kernel_ptr<__half, HD, 1, false, false, true>()))
        switch (head_dim) {
            case 64: return grid_for<64, false>(PA_GFN(64), s, num_kv_heads, max_context, ctas_override);
            case 128: return grid_for<128, false>(PA_GFN(128), s, num_kv_heads, max_context, ctas_override);
            default: return grid_for<256, false>(PA_GFN(256), s, num_kv_heads, max_context, ctas_override);
        }
#undef PA_GFN
    }
#define PA_KFN(HD, F8)                                                                                      \
    (bf ? (two ? kernel_ptr<__nv_bfloat16, HD, 2, F8>() : kernel_ptr<__nv_bfloat16, HD, 1, F8>())          \
        : (two ? kernel_ptr<__half, HD, 2, F8>() : kernel_ptr<__half, HD, 1, F8>()))
    if (kv_fp8) {
        if (head_dim == 128) return grid_for<128, true>(PA_KFN(128, true), s, num_kv_heads, max_context, ctas_override);
        return grid_for<256, true>(PA_KFN(256, true), s, num_kv_heads, max_context, ctas_override);
    }
    switch (head_dim) {
        case 64: return grid_for<64, false>(PA_KFN(64, false), s, num_kv_heads, max_context, ctas_override);
        case 128: return grid_for<128, false>(PA_KFN(128, false), s, num_kv_heads, max_context, ctas_override);
        default: return grid_for<256, false>(PA_KFN(256, false), s, num_kv_heads, max_context, ctas_override);
    }
#undef PA_KFN
}

int decode_tc_warps_per_cta(int32_t head_dim, bool kv_fp8) {
    if (kv_fp8) return head_dim == 256 ? Pipe<256, true>::NW : Pipe<128, true>::NW;
    return head_dim == 256 ? Pipe<256, false>::NW : (head_dim == 128 ? Pipe<128, false>::NW : Pipe<64, false>::NW);
}

size_t decode_tc_workspace(int32_t num_seqs, int32_t num_kv_heads, int32_t group, int32_t head_dim, int grid_ctas,
                           bool kv_fp8) {
    const int nw = decode_tc_warps_per_cta(head_dim, kv_fp8);
    return (size_t)grid_ctas * nw * 2 * group * (head_dim + 4) * sizeof(float);
}

cudaError_t launch_decode_tc(const AttnArgs& a, int32_t num_blocks, int grid_ctas, void* workspace,
                             std::string* err, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    return a.dtype == 1 ? launch_dtype<__nv_bfloat16>(a, num_blocks, grid_ctas, workspace, err, stream)
                        : launch_dtype<__half>(a, num_blocks, grid_ctas, workspace, err, stream);
}

uint32_t decode_tc_status(bool clear) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(v));
    if (clear) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_decode_status, &z, sizeof(z));
    }
    return v;
}

}  // namespace pa
