// pa_internal.h -- host-side declarations shared by the library's translation
// units (launchers called by the C ABI in pa_api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

namespace pa {

// Element size of a pa_dtype (PA_F32 = 0, PA_BF16 = 1, PA_F16 = 2, PA_FP8_E4M3 = 3).
inline int elt_size(int dtype) { return dtype == 0 ? 4 : (dtype == 3 ? 1 : 2); }

// Upper limit of sequences one tensor-core decode launch handles (its
// per-sequence block-count prefix lives in shared memory); the C ABI splits
// larger batches into launches of at most this many sequences.
constexpr int kDecodeMaxSeqsPerLaunch = 4096;

// Most layers one pa_copy_blocks call takes (their pointers travel in the
// kernel's parameter block).  Equal to PA_MAX_LAYERS of pa.h.
#define PA_MAX_LAYERS_INTERNAL 128

// Number of polls a bounded mbarrier wait makes before giving up.
constexpr uint32_t kMaxPolls = 1u << 24;

// Reason reported by pa_last_error() for the calling thread (pa_api.cu).
void record_error(const std::string& msg);

// Check mode (PA_OPT_CHECK_MODE) for entry points outside pa_api.cu: whether
// it is on, and the decode's index validation (lengths in [0, max_context],
// tables long enough, block ids in [0, num_blocks)) on host copies of the
// index arrays.  Returns a pa_status value (PA_OK, PA_ERR_INDEX or
// PA_ERR_CUDA) and records the reason for pa_last_error().
bool check_mode_on();
int check_decode_indices(const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                         int32_t num_seqs, int32_t num_blocks, int32_t block_size, int32_t max_context,
                         cudaStream_t stream);

// ---- copy kernels (pa_copy.cu)
cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_idx,
                                const int64_t* positions, int64_t n, int32_t block_size, int64_t* slot_out,
                                cudaStream_t stream);
cudaError_t launch_write_kv(const void* k, const void* v, const int64_t* slot_mapping, int64_t n, void* k_cache,
                            void* v_cache, int64_t row_bytes, cudaStream_t stream);
// Writes k_new[s] / v_new[s] ([S, Hkv, hd]) to each sequence's slot of
// position context_lens[s] - 1 (sequences with length 0 are skipped).
cudaError_t launch_append_kv(const void* k_new, const void* v_new, const int32_t* block_tables, int32_t max_blocks,
                             const int32_t* context_lens, int32_t num_seqs, int32_t block_size, void* k_cache,
                             void* v_cache, int64_t row_bytes, cudaStream_t stream);
cudaError_t launch_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k, void* const* dst_v,
                               int32_t num_layers, const int64_t* block_pairs, int32_t num_pairs, int64_t block_bytes,
                               cudaStream_t stream);
// Quantizing write: each (token, KV head) row of k / v ([n, Hkv, hd] of
// dtype) becomes E4M3 codes at its slot of k_codes / v_codes and one fp32
// scale in k_scales / v_scales [num_blocks, Hkv, block_size].
cudaError_t launch_write_kv_fp8(const void* k, const void* v, int dtype, const int64_t* slot_mapping, int64_t n,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, uint8_t* k_codes,
                                uint8_t* v_codes, float* k_scales, float* v_scales, cudaStream_t stream);
// The same for the generation step: sequence s's new rows go to the slot of
// position context_lens[s] - 1.
cudaError_t launch_append_kv_fp8(const void* k_new, const void* v_new, int dtype, const int32_t* block_tables,
                                 int32_t max_blocks, const int32_t* context_lens, int32_t num_seqs,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size, uint8_t* k_codes,
                                 uint8_t* v_codes, float* k_scales, float* v_scales, cudaStream_t stream);
cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                               const int64_t* block_pairs, int32_t num_pairs, int64_t block_bytes,
                               cudaStream_t stream);

// ---- CUDA-core attention (pa_attn_simt.cu): any dtype, head_dim <= 256.
// cu_seqlens_q == nullptr means one query per sequence (row i = sequence i).
struct AttnArgs {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    int32_t max_blocks;
    const int32_t* seq_lens;
    const int32_t* cu_seqlens_q;
    int32_t num_seqs;
    int32_t total_q;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    float scale;
    int causal;
    int dtype;
    // upper bound of seq_lens (varlen: sizes the work plan's buckets)
    int32_t max_context = 0;
    // decode only: the new token of each sequence (position L-1), written to
    // the pool and attended from these rows (nullptr: plain decode)
    const void* k_new = nullptr;
    const void* v_new = nullptr;
    // quantized cache: k_cache / v_cache hold E4M3 codes and these fp32
    // scales [num_blocks, num_kv_heads, block_size]; dtype is then the type
    // of q and out only
    int kv_fp8 = 0;
    const float* k_scales = nullptr;
    const float* v_scales = nullptr;
    // code cache, head_dim 128: the two tiles of a stage that belong to one
    // unit worked as one 32-token step
    int pair_steps = 0;
};
bool attn_simt_supported(int dtype, int head_dim);  // either cache kind
cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t stream);

// ---- tensor-core decode (pa_decode_tc.cu)
// kv_fp8: the cache holds E4M3 codes with scales (AttnArgs::kv_fp8).
bool decode_tc_supported(int dtype, int head_dim, int block_size, int group, bool kv_fp8 = false);
// Grid size (CTAs) the launch will use for this problem on the current device.
int decode_tc_grid(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                   int32_t max_context, int dtype, int32_t group, int64_t ctas_override, bool kv_fp8 = false);
int decode_tc_warps_per_cta(int32_t head_dim, bool kv_fp8 = false);
size_t decode_tc_workspace(int32_t num_seqs, int32_t num_kv_heads, int32_t group, int32_t head_dim, int grid_ctas,
                           bool kv_fp8 = false);
cudaError_t launch_decode_tc(const AttnArgs& a, int32_t num_blocks, int grid_ctas, void* workspace,
                             std::string* err, cudaStream_t stream);
uint32_t decode_tc_status(bool clear);
// ---- self-test of the failure path (pa_selftest.cu): one CTA waits on a
// barrier nothing completes for `polls` polls and sets its status word's
// timeout bit (pa_selftest_wait_timeout).
cudaError_t launch_selftest_wait(uint32_t polls, cudaStream_t stream);
uint32_t selftest_status(bool clear);

// ---- tcgen05 varlen (pa_varlen_umma.cu)
bool varlen_umma_supported(int dtype, int head_dim, int block_size, int group, bool kv_fp8 = false);
// Bytes of the optional workspace that lets the kernel run its work longest first.
size_t varlen_umma_workspace(int32_t num_seqs, int64_t total_q, int32_t group);
// workspace: nullptr (request order), or varlen_umma_workspace(...) bytes.
cudaError_t launch_varlen_umma(const AttnArgs& a, int32_t num_blocks, void* workspace, std::string* err,
                               cudaStream_t stream);
uint32_t varlen_umma_status(bool clear);

}  // namespace pa
