// pa_decode_noalloc.cu -- pa_decode_noalloc: the tensor-core decode with its
// scratch in a fixed device array owned by the library instead of a
// caller-supplied workspace.
//
// Who needs it: callers that must not allocate device memory at the time
// they run the decode -- an inference runtime or plugin host that owns all
// device memory through its own fixed pool and forbids cudaMalloc inside
// its execution callbacks, code on a latency-critical path where the device
// synchronisation an allocation can trigger is not acceptable, or a caller
// with no allocator handle at all.  They still pass q, the caches, tables,
// lengths and the output; only the split-KV scratch comes from here.
//
// The scratch is one file-scope array per device (kNoAllocScratchBytes,
// 8 MiB), present from module load until the process exits.  Its device
// address is looked up with cudaGetSymbolAddress on the first call made
// with that device current, and again whenever the device's context has
// changed since (after cudaDeviceReset the module is loaded afresh and the
// old address is gone); make that first call before any stream capture.
// Every call on a device shares the array, so two calls whose kernels
// overlap on the GPU (different streams without ordering) race on it.
// Nothing in it has to start at zero, and nothing a call leaves behind is
// read by a later one: each launch writes every split record its merge
// reads before the merge runs, and the merge finds them from the lengths.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address per device, with the id of the context it was
// looked up in.
struct ScratchSlot {
    void* addr = nullptr;
    unsigned long long ctx_id = 0;
};
std::mutex g_setup_mu;
ScratchSlot g_scratch[kMaxDevices];

pa_status noalloc_fail(pa_status st, const std::string& msg) {
    pa::record_error(msg);  // read back with pa_last_error()
    return st;
}

// Id of the calling thread's current context (0 if the driver cannot say).
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
        get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// Device address of this device's scratch array (looked up on first use,
// and again when the device's context has changed).
pa_status scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(PA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(PA_ERR_UNSUPPORTED, "device ordinal beyond 63");
    // Before the first runtime call that needs it, no context may be current
    // yet (id 0); the runtime makes the primary context current inside
    // cudaGetSymbolAddress, and the id is read again after it.
    std::lock_guard<std::mutex> lock(g_setup_mu);
    ScratchSlot& slot = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (slot.addr == nullptr || (id != 0 && id != slot.ctx_id)) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return noalloc_fail(PA_ERR_CUDA, std::string("cudaGetSymbolAddress of the scratch array: ") +
                                                 cudaGetErrorString(e));
        slot.addr = p;
        slot.ctx_id = current_context_id();
    }
    *out = slot.addr;
    return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                            int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t num_blocks, int32_t block_size, int32_t max_context, float scale, int dtype,
                            void* stream) {
    if (num_seqs < 0 || max_blocks < 0 || max_context < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || num_blocks <= 0 || block_size <= 0)
        return noalloc_fail(PA_ERR_INVALID_ARG, "sizes must be non-negative (head counts and dims positive)");
    if (num_heads % num_kv_heads != 0)
        return noalloc_fail(PA_ERR_INVALID_ARG, "num_heads must be a multiple of num_kv_heads");
    if ((int64_t)num_blocks * block_size > INT32_MAX)
        return noalloc_fail(PA_ERR_UNSUPPORTED, "num_blocks * block_size must fit in int32");
    const int G = num_heads / num_kv_heads;
    if (!pa::decode_tc_supported(dtype, head_dim, block_size, G))
        return noalloc_fail(PA_ERR_UNSUPPORTED, "pa_decode_noalloc takes bf16/f16, head_dim 64/128/256 and at "
                                                "most 16 query heads per KV head");
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return noalloc_fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return noalloc_fail(PA_ERR_INVALID_ARG, "out, q and the caches must be 16-byte aligned");

    const int grid = pa::decode_tc_grid(num_seqs, num_kv_heads, head_dim, block_size, max_context, dtype, G, 0);
    const size_t need = pa::decode_tc_workspace(num_seqs, num_kv_heads, G, head_dim, grid);
    if (need > kNoAllocScratchBytes)
        return noalloc_fail(PA_ERR_WORKSPACE, "this problem needs " + std::to_string(need) +
                                                  " bytes of scratch; pa_decode_noalloc holds at most " +
                                                  std::to_string(kNoAllocScratchBytes) +
                                                  " (use pa_decode with a workspace)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pa::check_mode_on()) {
        // host copies of the lengths and tables only; nothing on the device
        const int st = pa::check_decode_indices(block_tables, max_blocks, context_lens, num_seqs, num_blocks,
                                                block_size, max_context, s);
        if (st != PA_OK) return static_cast<pa_status>(st);
    }
    void* scratch = nullptr;
    pa_status st = scratch_for_current_device(&scratch);
    if (st != PA_OK) return st;

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
        std::string err;
        cudaError_t e = pa::launch_decode_tc(c, num_blocks, grid, scratch, &err, s);
        if (e != cudaSuccess)
            return noalloc_fail(PA_ERR_CUDA, "pa_decode_noalloc: " + (err.empty() ? std::string(cudaGetErrorString(e)) : err));
    }
    return PA_OK;
}

}  // extern "C"
