// pa_api.cu -- the extern "C" entry points declared in include/pa.h:
// argument validation, optional host-side index checking, and dispatch to
// the kernels' launchers.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <string>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

thread_local std::string g_last_error;
int64_t g_options[5] = {0, 0, 0, 0, 0};
constexpr int32_t kPairMinContext = 2048;  // automatic pair steps above this max_context

pa_status fail(pa_status st, const std::string& msg) {
    g_last_error = msg;
    return st;
}

pa_status cuda_fail(cudaError_t e, const char* where) {
    return fail(PA_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(int d) { return d == PA_F32 || d == PA_BF16 || d == PA_F16; }
cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

template <typename T>
bool to_host(std::vector<T>& dst, const T* src, int64_t n, cudaStream_t st, pa_status* err) {
    dst.resize((size_t)std::max<int64_t>(n, 0));
    if (n <= 0) return true;
    cudaError_t e = cudaMemcpyAsync(dst.data(), src, sizeof(T) * (size_t)n, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        *err = cuda_fail(e, "check mode: copying indices to the host");
        return false;
    }
    return true;
}

bool check_mode() { return g_options[PA_OPT_CHECK_MODE] != 0; }

// Check-mode validation of block tables against lengths.
pa_status check_tables(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks, const std::vector<int32_t>& lens,
                       int32_t num_blocks, int32_t block_size, int32_t max_context, cudaStream_t st) {
    pa_status err = PA_OK;
    std::vector<int32_t> bt;
    if (!to_host(bt, block_tables, (int64_t)num_seqs * max_blocks, st, &err)) return err;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t L = lens[s];
        if (L < 0 || L > max_context)
            return fail(PA_ERR_INDEX, "sequence " + std::to_string(s) + ": length " + std::to_string(L) +
                                          " outside [0, max_context=" + std::to_string(max_context) + "]");
        const int64_t nb = ((int64_t)L + block_size - 1) / block_size;
        if (nb > max_blocks)
            return fail(PA_ERR_INDEX, "sequence " + std::to_string(s) + " needs " + std::to_string(nb) +
                                          " blocks but the table holds " + std::to_string(max_blocks));
        for (int64_t b = 0; b < nb; ++b) {
            const int32_t id = bt[(size_t)s * max_blocks + b];
            if (id < 0 || id >= num_blocks)
                return fail(PA_ERR_INDEX, "sequence " + std::to_string(s) + " logical block " + std::to_string(b) +
                                              " maps to " + std::to_string(id) + ", outside [0, num_blocks)");
        }
    }
    return PA_OK;
}

// bytes_only: the call moves bytes (copy, swap), so PA_FP8_E4M3 pools are
// accepted as well.
pa_status check_geometry(int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                         int32_t block_size, int dtype, bool bytes_only = false) {
    if (!valid_dtype(dtype) && !(bytes_only && dtype == PA_FP8_E4M3))
        return fail(PA_ERR_INVALID_ARG, bytes_only ? "dtype must be PA_F32, PA_BF16, PA_F16 or PA_FP8_E4M3"
                                                   : "dtype must be PA_F32, PA_BF16 or PA_F16");
    if (num_kv_heads <= 0 || num_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || block_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "head counts, head_dim, num_blocks and block_size must be positive");
    if (num_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_heads must be a multiple of num_kv_heads");
    if ((int64_t)num_blocks * block_size > INT32_MAX)
        return fail(PA_ERR_UNSUPPORTED, "num_blocks * block_size must fit in int32");
    return PA_OK;
}

// Check-mode validation of a slot mapping: in the pool, or negative (skip); distinct.
pa_status check_slots(const int64_t* slot_mapping, int64_t n, int32_t num_blocks, int32_t block_size,
                      cudaStream_t st) {
    pa_status err = PA_OK;
    std::vector<int64_t> sm;
    if (!to_host(sm, slot_mapping, n, st, &err)) return err;
    const int64_t slots = (int64_t)num_blocks * block_size;
    std::unordered_set<int64_t> seen;
    for (int64_t i = 0; i < n; ++i) {
        if (sm[i] < 0) continue;
        if (sm[i] >= slots)
            return fail(PA_ERR_INDEX, "token " + std::to_string(i) + ": slot " + std::to_string(sm[i]) +
                                          " outside the pool");
        if (!seen.insert(sm[i]).second)
            return fail(PA_ERR_INDEX, "slot " + std::to_string(sm[i]) + " written twice in one call");
    }
    return PA_OK;
}

}  // namespace

namespace pa {
// Sets the reason pa_last_error() reports (used by entry points defined in
// other translation units).
void record_error(const std::string& msg) { g_last_error = msg; }

bool check_mode_on() { return check_mode(); }

int check_decode_indices(const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                         int32_t num_seqs, int32_t num_blocks, int32_t block_size, int32_t max_context,
                         cudaStream_t stream) {
    pa_status err = PA_OK;
    std::vector<int32_t> lens;
    if (!to_host(lens, context_lens, num_seqs, stream, &err)) return err;
    return check_tables(block_tables, num_seqs, max_blocks, lens, num_blocks, block_size, max_context, stream);
}
}  // namespace pa

extern "C" {

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_INDEX: return "PA_ERR_INDEX";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        default: return "unknown pa_status";
    }
}

const char* pa_last_error(void) { return g_last_error.c_str(); }

pa_status pa_set_option(int option, int64_t value) {
    if (option < 0 || option > PA_OPT_FP8_PAIR_STEP) return fail(PA_ERR_INVALID_ARG, "unknown option");
    if ((option == PA_OPT_DECODE_KERNEL && value > 2) || (option == PA_OPT_VARLEN_KERNEL && value > 2) ||
        (option == PA_OPT_FP8_PAIR_STEP && value > 2))
        return fail(PA_ERR_INVALID_ARG, "unknown kernel choice");
    if (value < 0) return fail(PA_ERR_INVALID_ARG, "option values are non-negative");
    g_options[option] = value;
    return PA_OK;
}

int64_t pa_get_option(int option) {
    if (option < 0 || option > PA_OPT_FP8_PAIR_STEP) return -1;
    return g_options[option];
}

pa_status pa_set_check_mode(int on) { return pa_set_option(PA_OPT_CHECK_MODE, on ? 1 : 0); }

pa_status pa_device_status(int clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "pa_device_status");
    const uint32_t bits =
        pa::decode_tc_status(clear != 0) | pa::varlen_umma_status(clear != 0) | pa::selftest_status(clear != 0);
    if (bits & 1u) return fail(PA_ERR_TIMEOUT, "a kernel's bounded barrier wait ran out");
    return PA_OK;
}

pa_status pa_selftest_wait_timeout(int32_t polls, void* stream) {
    if (polls < 1 || polls > (1 << 20)) return fail(PA_ERR_INVALID_ARG, "polls must be in [1, 2^20]");
    cudaError_t e = pa::launch_selftest_wait((uint32_t)polls, as_stream(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_selftest_wait_timeout launch");
}

pa_status pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks, const int32_t* seq_idx,
                          const int64_t* positions, int64_t n, int32_t block_size, int64_t* slot_out,
                          void* stream) {
    if (n < 0 || num_seqs < 0 || max_blocks < 0 || block_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "sizes must be non-negative and block_size positive");
    if (n == 0) return PA_OK;
    if (!block_tables || !seq_idx || !positions || !slot_out) return fail(PA_ERR_INVALID_ARG, "null pointer");
    cudaStream_t st = as_stream(stream);
    if (check_mode()) {
        pa_status err = PA_OK;
        std::vector<int32_t> si;
        std::vector<int64_t> pos;
        if (!to_host(si, seq_idx, n, st, &err) || !to_host(pos, positions, n, st, &err)) return err;
        for (int64_t i = 0; i < n; ++i) {
            if (pos[i] < 0) continue;
            if (si[i] < 0 || si[i] >= num_seqs)
                return fail(PA_ERR_INDEX, "token " + std::to_string(i) + ": sequence index out of range");
            if (pos[i] / block_size >= max_blocks)
                return fail(PA_ERR_INDEX, "token " + std::to_string(i) + ": position beyond the block table");
        }
    }
    cudaError_t e = pa::launch_slot_mapping(block_tables, max_blocks, seq_idx, positions, n, block_size, slot_out, st);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_slot_mapping launch");
}

pa_status pa_write_kv(const void* k, const void* v, const int64_t* slot_mapping, int64_t n, void* k_cache,
                      void* v_cache, int32_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                      int dtype, void* stream) {
    pa_status g = check_geometry(num_kv_heads, num_kv_heads, head_dim, num_blocks, block_size, dtype);
    if (g != PA_OK) return g;
    if (n < 0) return fail(PA_ERR_INVALID_ARG, "n must be non-negative");
    if (n == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return fail(PA_ERR_INVALID_ARG, "null pointer");
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * pa::elt_size(dtype);
    if (row_bytes % 16 != 0)
        return fail(PA_ERR_UNSUPPORTED, "num_kv_heads * head_dim * element size must be a multiple of 16 bytes");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "k, v and the caches must be 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    if (check_mode()) {
        pa_status err = check_slots(slot_mapping, n, num_blocks, block_size, st);
        if (err != PA_OK) return err;
    }
    cudaError_t e = pa::launch_write_kv(k, v, slot_mapping, n, k_cache, v_cache, row_bytes, st);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_write_kv launch");
}

pa_status pa_write_kv_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t n, void* k_codes,
                          void* v_codes, float* k_scales, float* v_scales, int32_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim, int dtype, void* stream) {
    pa_status g = check_geometry(num_kv_heads, num_kv_heads, head_dim, num_blocks, block_size, dtype);
    if (g != PA_OK) return g;
    if (head_dim > 256) return fail(PA_ERR_UNSUPPORTED, "head_dim must be at most 256");
    if (n < 0) return fail(PA_ERR_INVALID_ARG, "n must be non-negative");
    if (n == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_codes || !v_codes || !k_scales || !v_scales)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_codes) || !aligned16(v_codes))
        return fail(PA_ERR_INVALID_ARG, "k, v and the code pools must be 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    if (check_mode()) {
        pa_status err = check_slots(slot_mapping, n, num_blocks, block_size, st);
        if (err != PA_OK) return err;
    }
    cudaError_t e = pa::launch_write_kv_fp8(k, v, dtype, slot_mapping, n, num_kv_heads, head_dim, block_size,
                                            static_cast<uint8_t*>(k_codes), static_cast<uint8_t*>(v_codes), k_scales,
                                            v_scales, st);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_write_kv_fp8 launch");
}

pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers, const int64_t* block_pairs,
                         int32_t num_pairs, int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim, int dtype, void* stream) {
    pa_status g = check_geometry(num_kv_heads, num_kv_heads, head_dim, num_blocks, block_size, dtype, true);
    if (g != PA_OK) return g;
    if (num_pairs < 0) return fail(PA_ERR_INVALID_ARG, "num_pairs must be non-negative");
    if (num_layers < 1 || num_layers > PA_MAX_LAYERS)
        return fail(PA_ERR_INVALID_ARG, "num_layers must be in [1, PA_MAX_LAYERS]");
    if (num_pairs == 0) return PA_OK;
    if (!k_caches || !v_caches || !block_pairs) return fail(PA_ERR_INVALID_ARG, "null pointer");
    for (int l = 0; l < num_layers; ++l) {
        if (!k_caches[l] || !v_caches[l]) return fail(PA_ERR_INVALID_ARG, "null cache pointer");
        if (!aligned16(k_caches[l]) || !aligned16(v_caches[l]))
            return fail(PA_ERR_INVALID_ARG, "caches must be 16-byte aligned");
    }
    const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_dim * pa::elt_size(dtype);
    if (block_bytes % 16 != 0) return fail(PA_ERR_UNSUPPORTED, "a block must be a multiple of 16 bytes");
    cudaStream_t st = as_stream(stream);
    if (check_mode()) {
        pa_status err = PA_OK;
        std::vector<int64_t> pr;
        if (!to_host(pr, block_pairs, 2 * (int64_t)num_pairs, st, &err)) return err;
        std::unordered_set<int64_t> dsts, srcs;
        for (int32_t p = 0; p < num_pairs; ++p) {
            const int64_t s = pr[2 * p], d = pr[2 * p + 1];
            if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks)
                return fail(PA_ERR_INDEX, "pair " + std::to_string(p) + ": block id outside [0, num_blocks)");
            if (!dsts.insert(d).second)
                return fail(PA_ERR_INDEX, "block " + std::to_string(d) + " is the destination of two pairs");
            srcs.insert(s);
        }
        for (int32_t p = 0; p < num_pairs; ++p) {
            const int64_t s = pr[2 * p], d = pr[2 * p + 1];
            if (d != s && srcs.count(d))
                return fail(PA_ERR_INDEX, "block " + std::to_string(d) + " is both a destination and a source");
        }
    }
    cudaError_t e = pa::launch_copy_blocks(k_caches, v_caches, num_layers, block_pairs, num_pairs, block_bytes, st);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_copy_blocks launch");
}

// Device address a kernel can use for p: device memory as is, pinned or
// registered host memory through its device mapping; nullptr otherwise.
static const void* device_view(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
    if (at.type == cudaMemoryTypeHost && at.devicePointer) {
        const uint8_t* base = static_cast<const uint8_t*>(at.hostPointer);
        return static_cast<const uint8_t*>(at.devicePointer) + (static_cast<const uint8_t*>(p) - base);
    }
    return nullptr;
}

pa_status pa_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k, void* const* dst_v,
                         int32_t num_layers, const int64_t* block_pairs, int32_t num_pairs, int32_t src_num_blocks,
                         int32_t dst_num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int dtype,
                         void* stream) {
    if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "num_pairs must be non-negative and both pools non-empty");
    pa_status g = check_geometry(num_kv_heads, num_kv_heads, head_dim, src_num_blocks, block_size, dtype, true);
    if (g != PA_OK) return g;
    if (num_layers < 1 || num_layers > PA_MAX_LAYERS)
        return fail(PA_ERR_INVALID_ARG, "num_layers must be in [1, PA_MAX_LAYERS]");
    if (num_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !block_pairs) return fail(PA_ERR_INVALID_ARG, "null pointer");
    const int64_t block_bytes = (int64_t)block_size * num_kv_heads * head_dim * pa::elt_size(dtype);
    if (block_bytes % 16 != 0) return fail(PA_ERR_UNSUPPORTED, "a block must be a multiple of 16 bytes");
    std::vector<void*> sk(num_layers), sv(num_layers), dk(num_layers), dv(num_layers);
    for (int l = 0; l < num_layers; ++l) {
        const void* in[4] = {src_k[l], src_v[l], dst_k[l], dst_v[l]};
        void** out[4] = {&sk[l], &sv[l], &dk[l], &dv[l]};
        for (int i = 0; i < 4; ++i) {
            if (!in[i] || !aligned16(in[i])) return fail(PA_ERR_INVALID_ARG, "pools must be non-null and 16-byte aligned");
            const void* d = device_view(in[i]);
            if (!d)
                return fail(PA_ERR_INVALID_ARG, "a pool is neither device memory nor pinned/registered host memory");
            *out[i] = const_cast<void*>(d);
        }
    }
    const void* pairs_dev = device_view(block_pairs);
    if (!pairs_dev) return fail(PA_ERR_INVALID_ARG, "block_pairs must be device or pinned host memory");
    cudaStream_t st = as_stream(stream);
    if (check_mode()) {
        pa_status err = PA_OK;
        std::vector<int64_t> pr;
        if (!to_host(pr, static_cast<const int64_t*>(pairs_dev), 2 * (int64_t)num_pairs, st, &err)) return err;
        std::unordered_set<int64_t> dsts;
        for (int32_t p = 0; p < num_pairs; ++p) {
            const int64_t s = pr[2 * p], d = pr[2 * p + 1];
            if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks)
                return fail(PA_ERR_INDEX, "pair " + std::to_string(p) + ": block id outside its pool");
            if (!dsts.insert(d).second)
                return fail(PA_ERR_INDEX, "block " + std::to_string(d) + " is the destination of two pairs");
        }
    }
    cudaError_t e = pa::launch_swap_blocks(sk.data(), sv.data(), dk.data(), dv.data(), num_layers,
                                           static_cast<const int64_t*>(pairs_dev), num_pairs, block_bytes, st);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_swap_blocks launch");
}

// ------------------------------------------------------------------ decode

static bool use_decode_tc(int dtype, int head_dim, int block_size, int group, bool kv_fp8, pa_status* st) {
    const int64_t want = g_options[PA_OPT_DECODE_KERNEL];
    const bool ok = pa::decode_tc_supported(dtype, head_dim, block_size, group, kv_fp8);
    *st = PA_OK;
    if (want == 1) return false;
    if (want == 2 && !ok) {
        *st = fail(PA_ERR_UNSUPPORTED, kv_fp8 ? "the tensor-core decode kernel over an FP8 cache takes bf16/f16 "
                                                "queries, head_dim 128/256, block_size 8 or a multiple of 16 up "
                                                "to 256, and at most 16 query heads per KV head"
                                              : "the tensor-core decode kernel takes bf16/f16, head_dim 64/128/256 "
                                                "and at most 16 query heads per KV head");
        return false;
    }
    return ok;
}

static size_t decode_workspace(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t max_context, int dtype, bool kv_fp8) {
    if (num_seqs <= 0 || num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads || max_context < 0)
        return 0;
    pa_status st;
    const int G = num_heads / num_kv_heads;
    if (!use_decode_tc(dtype, head_dim, block_size, G, kv_fp8, &st)) return 0;
    const int grid = pa::decode_tc_grid(num_seqs, num_kv_heads, head_dim, block_size, max_context, dtype, G,
                                        g_options[PA_OPT_DECODE_CTAS], kv_fp8);
    return pa::decode_tc_workspace(num_seqs, num_kv_heads, G, head_dim, grid, kv_fp8);
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, int32_t max_context, int dtype) {
    return decode_workspace(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context, dtype, false);
}

size_t pa_decode_fp8_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t max_context, int dtype) {
    return decode_workspace(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context, dtype, true);
}

}  // extern "C"

// k_scales != nullptr: the caches hold E4M3 codes with these scales.
static pa_status decode_impl(void* out, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                             const void* v_cache, const float* k_scales, const float* v_scales,
                             const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                             int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t num_blocks, int32_t block_size, int32_t max_context, float scale, int dtype,
                             void* workspace, size_t workspace_bytes, void* stream) {
    const bool fp8 = k_scales != nullptr;
    pa_status g = check_geometry(num_heads, num_kv_heads, head_dim, num_blocks, block_size, dtype);
    if (g != PA_OK) return g;
    if (num_seqs < 0 || max_blocks < 0 || max_context < 0)
        return fail(PA_ERR_INVALID_ARG, "num_seqs, max_blocks and max_context must be non-negative");
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    const bool append = k_new != nullptr || v_new != nullptr;
    if (append && (!k_new || !v_new)) return fail(PA_ERR_INVALID_ARG, "k_new and v_new go together");
    if (append && (!aligned16(k_new) || !aligned16(v_new)))
        return fail(PA_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (append && ((int64_t)num_kv_heads * head_dim * pa::elt_size(dtype)) % 16 != 0)
        return fail(PA_ERR_UNSUPPORTED, "num_kv_heads * head_dim * element size must be a multiple of 16 bytes");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "out, q and the caches must be 16-byte aligned");
    if (!pa::attn_simt_supported(dtype, head_dim)) return fail(PA_ERR_UNSUPPORTED, "head_dim must be in [1, 256]");
    if (fp8 && (!v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
        return fail(PA_ERR_INVALID_ARG, "k_scales and v_scales must be non-null and 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    if (check_mode()) {
        pa_status err = PA_OK;
        std::vector<int32_t> lens;
        if (!to_host(lens, context_lens, num_seqs, st, &err)) return err;
        err = check_tables(block_tables, num_seqs, max_blocks, lens, num_blocks, block_size, max_context, st);
        if (err != PA_OK) return err;
    }
    pa::AttnArgs a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks;
    a.seq_lens = context_lens;
    a.cu_seqlens_q = nullptr;
    a.num_seqs = num_seqs;
    a.total_q = num_seqs;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.scale = scale;
    a.causal = 1;
    a.dtype = dtype;
    a.kv_fp8 = fp8 ? 1 : 0;
    a.k_scales = k_scales;
    a.v_scales = v_scales;

    const int G = num_heads / num_kv_heads;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * pa::elt_size(dtype);
    pa_status sel;
    const bool tc = use_decode_tc(dtype, head_dim, block_size, G, fp8, &sel);
    if (sel != PA_OK) return sel;
    // The tensor-core kernel fuses the append for 16-bit caches, and for code
    // caches of head_dim 128 when the batch has no more (sequence, KV head)
    // units than the grid has warps: quantizing inside the kernel costs the
    // warp that owns a unit's last tile some microseconds (measured: a gain
    // with 512 units on 1,824 warps, a loss with 5,120), while a separate
    // quantizing kernel spreads the rows over the whole GPU.  Otherwise the
    // new rows are written (quantized for a code cache) by a separate kernel
    // first, then attended from the pool; either way the pool and the output
    // are the same bit for bit.
    bool fused_append = append && tc && (!fp8 || head_dim == 128);
    if (fused_append && fp8) {
        const int64_t warps = (int64_t)pa::decode_tc_grid(num_seqs, num_kv_heads, head_dim, block_size, max_context,
                                                          dtype, G, g_options[PA_OPT_DECODE_CTAS], fp8) *
                              pa::decode_tc_warps_per_cta(head_dim, fp8);
        fused_append = (int64_t)num_seqs * num_kv_heads <= warps;
    }
    if (append && !fused_append) {
        cudaError_t e = fp8 ? pa::launch_append_kv_fp8(k_new, v_new, dtype, block_tables, max_blocks, context_lens,
                                                       num_seqs, num_kv_heads, head_dim, block_size,
                                                       static_cast<uint8_t*>(const_cast<void*>(k_cache)),
                                                       static_cast<uint8_t*>(const_cast<void*>(v_cache)),
                                                       const_cast<float*>(k_scales), const_cast<float*>(v_scales), st)
                            : pa::launch_append_kv(k_new, v_new, block_tables, max_blocks, context_lens, num_seqs,
                                                   block_size, const_cast<void*>(k_cache),
                                                   const_cast<void*>(v_cache), row_bytes, st);
        if (e != cudaSuccess) return cuda_fail(e, "pa_decode_append launch");
    }
    if (!tc) {
        cudaError_t e = pa::launch_attn_simt(a, st);
        return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_decode launch");
    }
    const int grid = pa::decode_tc_grid(num_seqs, num_kv_heads, head_dim, block_size, max_context, dtype, G,
                                        g_options[PA_OPT_DECODE_CTAS], fp8);
    const size_t need = pa::decode_tc_workspace(num_seqs, num_kv_heads, G, head_dim, grid, fp8);
    // Code cache, head_dim 128: the 32-token pair step pays where units are
    // long (measured: 8 x 32k tokens 7 % faster, the 64-sequence batch of up
    // to 3,360 tokens 1 %) and loses where many units are short (128
    // sequences of mean 480 tokens: 8 % slower, the split then leaves some
    // warps with many single tiles).  max_context is the host's only view
    // of the lengths.
    const int64_t pair_opt = g_options[PA_OPT_FP8_PAIR_STEP];
    a.pair_steps = fp8 && head_dim == 128 && (pair_opt == 2 || (pair_opt == 0 && max_context > kPairMinContext));
    if (workspace_bytes < need || (need && !workspace))
        return fail(PA_ERR_WORKSPACE, "workspace holds " + std::to_string(workspace_bytes) + " bytes, " +
                                          std::to_string(need) + " needed");
    if (!aligned16(workspace)) return fail(PA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    const int64_t elt = pa::elt_size(dtype);
    for (int32_t s0 = 0; s0 < num_seqs; s0 += pa::kDecodeMaxSeqsPerLaunch) {
        pa::AttnArgs c = a;
        const int32_t cnt = std::min(num_seqs - s0, pa::kDecodeMaxSeqsPerLaunch);
        c.num_seqs = cnt;
        c.total_q = cnt;
        c.out = static_cast<uint8_t*>(out) + (int64_t)s0 * num_heads * head_dim * elt;
        c.q = static_cast<const uint8_t*>(q) + (int64_t)s0 * num_heads * head_dim * elt;
        c.block_tables = block_tables + (int64_t)s0 * max_blocks;
        c.seq_lens = context_lens + s0;
        if (fused_append) {
            c.k_new = static_cast<const uint8_t*>(k_new) + (int64_t)s0 * row_bytes;
            c.v_new = static_cast<const uint8_t*>(v_new) + (int64_t)s0 * row_bytes;
        }
        std::string err;
        cudaError_t e = pa::launch_decode_tc(c, num_blocks, grid, workspace, &err, st);
        if (e != cudaSuccess)
            return err.empty() ? cuda_fail(e, "pa_decode launch") : fail(PA_ERR_CUDA, "pa_decode: " + err);
    }
    return PA_OK;
}

extern "C" {

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                    int32_t max_blocks, const int32_t* context_lens, int32_t num_seqs, int32_t num_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                    int32_t max_context, float scale, int dtype, void* workspace, size_t workspace_bytes,
                    void* stream) {
    return decode_impl(out, q, nullptr, nullptr, k_cache, v_cache, nullptr, nullptr, block_tables, max_blocks,
                       context_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_context,
                       scale, dtype, workspace, workspace_bytes, stream);
}

pa_status pa_decode_fp8(void* out, const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
                        const float* v_scales, const int32_t* block_tables, int32_t max_blocks,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t num_blocks, int32_t block_size, int32_t max_context, float scale,
                        int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs > 0 && (!k_scales || !v_scales)) return fail(PA_ERR_INVALID_ARG, "null pointer");
    return decode_impl(out, q, nullptr, nullptr, k_codes, v_codes, k_scales, v_scales, block_tables, max_blocks,
                       context_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_context,
                       scale, dtype, workspace, workspace_bytes, stream);
}

pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
                           void* v_cache, const int32_t* block_tables, int32_t max_blocks,
                           const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t num_blocks, int32_t block_size, int32_t max_context,
                           float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new)) return fail(PA_ERR_INVALID_ARG, "null pointer");
    return decode_impl(out, q, k_new, v_new, k_cache, v_cache, nullptr, nullptr, block_tables, max_blocks,
                       context_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_context,
                       scale, dtype, workspace, workspace_bytes, stream);
}

pa_status pa_decode_append_fp8(void* out, const void* q, const void* k_new, const void* v_new, void* k_codes,
                               void* v_codes, float* k_scales, float* v_scales, const int32_t* block_tables,
                               int32_t max_blocks, const int32_t* context_lens, int32_t num_seqs, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                               int32_t max_context, float scale, int dtype, void* workspace, size_t workspace_bytes,
                               void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new || !k_scales || !v_scales)) return fail(PA_ERR_INVALID_ARG, "null pointer");
    return decode_impl(out, q, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_tables, max_blocks,
                       context_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks, block_size, max_context,
                       scale, dtype, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------ varlen

size_t pa_varlen_workspace_size(int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t max_context,
                                int dtype) {
    (void)max_q, (void)max_context;
    if (num_seqs <= 0 || total_q <= 0 || num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads) return 0;
    const int G = num_heads / num_kv_heads;
    const int64_t want = g_options[PA_OPT_VARLEN_KERNEL];
    if (want == 1 || !pa::varlen_umma_supported(dtype, head_dim, block_size, G)) return 0;
    return pa::varlen_umma_workspace(num_seqs, total_q, G);
}

}  // extern "C"

// k_scales != nullptr: the caches hold E4M3 codes with these scales.
static pa_status varlen_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const float* k_scales, const float* v_scales, const int32_t* block_tables,
                             int32_t max_blocks, const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                             int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                             int32_t max_context, float scale, int causal, int dtype, void* workspace,
                             size_t workspace_bytes, void* stream) {
    const bool fp8 = k_scales != nullptr;
    pa_status g = check_geometry(num_heads, num_kv_heads, head_dim, num_blocks, block_size, dtype);
    if (g != PA_OK) return g;
    if (num_seqs < 0 || total_q < 0 || max_q < 0 || max_blocks < 0 || max_context < 0)
        return fail(PA_ERR_INVALID_ARG, "sizes must be non-negative");
    if (num_seqs == 0 || total_q == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !cu_seqlens_q)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "out, q and the caches must be 16-byte aligned");
    if (fp8 && (!v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
        return fail(PA_ERR_INVALID_ARG, "k_scales and v_scales must be non-null and 16-byte aligned");
    if (!pa::attn_simt_supported(dtype, head_dim)) return fail(PA_ERR_UNSUPPORTED, "head_dim must be in [1, 256]");
    const bool um_ok = pa::varlen_umma_supported(dtype, head_dim, block_size, num_heads / num_kv_heads, fp8);
    const int64_t want = g_options[PA_OPT_VARLEN_KERNEL];
    if (want == 2 && !um_ok)
        return fail(PA_ERR_UNSUPPORTED, fp8 ? "the tcgen05 varlen kernel over a code cache takes bf16/f16 "
                                              "queries, head_dim 128 and block_size 8 or a multiple of 16"
                                            : "the tcgen05 varlen kernel takes bf16/f16, head_dim 64/128/256 and "
                                              "block_size a multiple of 16 (or 8, below head_dim 256)");
    const bool use_um = um_ok && (want == 2 || want == 0);
    cudaStream_t st = as_stream(stream);
    if (check_mode()) {
        pa_status err = PA_OK;
        std::vector<int32_t> lens, cu;
        if (!to_host(lens, seq_lens, num_seqs, st, &err) || !to_host(cu, cu_seqlens_q, num_seqs + 1, st, &err))
            return err;
        if (cu[0] != 0 || cu[num_seqs] != total_q)
            return fail(PA_ERR_INDEX, "cu_seqlens_q must start at 0 and end at total_q");
        for (int32_t i = 0; i < num_seqs; ++i) {
            const int32_t nn = cu[i + 1] - cu[i];
            if (nn < 0) return fail(PA_ERR_INDEX, "cu_seqlens_q must be non-decreasing");
            if (nn > max_q) return fail(PA_ERR_INDEX, "request " + std::to_string(i) + " has more than max_q queries");
            if (nn > lens[i])
                return fail(PA_ERR_INDEX, "request " + std::to_string(i) + " has more new tokens than context");
        }
        err = check_tables(block_tables, num_seqs, max_blocks, lens, num_blocks, block_size, max_context, st);
        if (err != PA_OK) return err;
    }
    pa::AttnArgs a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks;
    a.seq_lens = seq_lens;
    a.cu_seqlens_q = cu_seqlens_q;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.dtype = dtype;
    a.max_context = max_context;
    a.kv_fp8 = fp8 ? 1 : 0;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    if (use_um) {
        // optional workspace: the tensor-core kernel then runs its work
        // longest first (a plan kernel sorts it); without one, in request order
        void* ws = nullptr;
        if (workspace && workspace_bytes > 0) {
            const size_t need = pa::varlen_umma_workspace(num_seqs, total_q, num_heads / num_kv_heads);
            if (workspace_bytes < need)
                return fail(PA_ERR_WORKSPACE, "workspace holds " + std::to_string(workspace_bytes) + " bytes, " +
                                                  std::to_string(need) + " needed");
            if (!aligned16(workspace)) return fail(PA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
            ws = workspace;
        }
        std::string err;
        cudaError_t e = pa::launch_varlen_umma(a, num_blocks, ws, &err, st);
        if (e != cudaSuccess)
            return err.empty() ? cuda_fail(e, "pa_varlen launch") : fail(PA_ERR_CUDA, "pa_varlen: " + err);
        return PA_OK;
    }
    cudaError_t e = pa::launch_attn_simt(a, st);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "pa_varlen launch");
}

extern "C" {

pa_status pa_varlen(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                    int32_t max_blocks, const int32_t* seq_lens, const int32_t* cu_seqlens_q, int32_t num_seqs,
                    int32_t total_q, int32_t max_q, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t num_blocks, int32_t block_size, int32_t max_context, float scale, int causal, int dtype,
                    void* workspace, size_t workspace_bytes, void* stream) {
    return varlen_impl(out, q, k_cache, v_cache, nullptr, nullptr, block_tables, max_blocks, seq_lens, cu_seqlens_q,
                       num_seqs, total_q, max_q, num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                       max_context, scale, causal, dtype, workspace, workspace_bytes, stream);
}

size_t pa_varlen_fp8_workspace_size(int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                    int32_t max_context, int dtype) {
    (void)max_q, (void)max_context;
    if (num_seqs <= 0 || total_q <= 0 || num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads) return 0;
    const int G = num_heads / num_kv_heads;
    if (g_options[PA_OPT_VARLEN_KERNEL] == 1 || !pa::varlen_umma_supported(dtype, head_dim, block_size, G, true))
        return 0;
    return pa::varlen_umma_workspace(num_seqs, total_q, G);
}

pa_status pa_varlen_fp8(void* out, const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
                        const float* v_scales, const int32_t* block_tables, int32_t max_blocks,
                        const int32_t* seq_lens, const int32_t* cu_seqlens_q, int32_t num_seqs, int32_t total_q,
                        int32_t max_q, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                        int32_t block_size, int32_t max_context, float scale, int causal, int dtype, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (num_seqs > 0 && total_q > 0 && (!k_scales || !v_scales)) return fail(PA_ERR_INVALID_ARG, "null pointer");
    return varlen_impl(out, q, k_codes, v_codes, k_scales, v_scales, block_tables, max_blocks, seq_lens,
                       cu_seqlens_q, num_seqs, total_q, max_q, num_heads, num_kv_heads, head_dim, num_blocks,
                       block_size, max_context, scale, causal, dtype, workspace, workspace_bytes, stream);
}

}  // extern "C"
