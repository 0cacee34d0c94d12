// pa_static_ws.cu -- pa_decode_static_workspace: the v2 path with its
// partition workspace in a fixed device array owned by this library, for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running inside a memory pool or
// allocator that must not re-enter the CUDA allocator, plug-ins whose host
// application owns every device allocation, or code that must not allocate
// between set-up and shutdown.  For them this entry point keeps the per-call
// scratch of the two-kernel (v2) path -- exp_sums, max_logits and tmp_out --
// in one file-scope __device__ array instead of caller-provided buffers.
//
// Properties a user must know:
//  * The array holds PA_STATIC_WORKSPACE_FLOATS floats (16 MiB).  Every GPU on
//    which the library's device code is loaded keeps it until the process exits.
//  * The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
//  * Every call on a device uses the same array and leaves its contents behind
//    for the next call.  Calls whose kernels overlap on the GPU (different
//    streams without ordering) race on it and give wrong results.
//  * Nothing in the array needs to start at zero: each entry a call reads was
//    written earlier in that call.
//  * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
#include <cuda_runtime.h>

#include <mutex>

#include "pa_decode.h"

namespace {

static __device__ __align__(256) float g_static_workspace[PA_STATIC_WORKSPACE_FLOATS];

constexpr int kMaxDevices = 64;

// Device address of g_static_workspace on the current device, looked up once
// per device with that device current.
float* static_workspace_address() {
    static std::mutex mu;
    static float* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        float* p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_static_workspace) != cudaSuccess)
            return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" pa_status pa_decode_static_workspace(const pa_decode_args* args, void* stream) {
    if (!args) return PA_ERR_INVALID_ARG;
    if (args->num_seqs < 0 || args->num_heads <= 0 || args->head_size <= 0 || args->max_seq_len < 0)
        return PA_ERR_INVALID_ARG;
    // workspace rows: one per query token (one per sequence without query_start)
    const int64_t rows = args->query_start ? args->num_query_tokens : args->num_seqs;
    if (rows < 0) return PA_ERR_INVALID_ARG;
    // rows * num_heads * P * (head_size + 2) <= capacity, checked factor by
    // factor so that no product of the (int32) sizes can wrap: each partial
    // product stays below the capacity (2^22) times an int32.
    const int64_t cap = PA_STATIC_WORKSPACE_FLOATS;
    const int64_t per_stat = (int64_t)args->head_size + 2;  // floats per (row, head, partition)
    const int64_t parts = pa_max_num_partitions(args->max_seq_len);
    if (rows > cap / args->num_heads) return PA_ERR_WORKSPACE;
    const int64_t row_heads = rows * args->num_heads;  // <= cap
    if (parts > cap / per_stat) return PA_ERR_WORKSPACE;
    if (row_heads > 0 && parts * per_stat > cap / row_heads) return PA_ERR_WORKSPACE;
    const int64_t stats = row_heads * parts;
    // tmp_out first (16-byte alignment for its float4 accesses), then the two statistics arrays
    const int64_t tmp = stats * args->head_size;
    if (args->num_seqs == 0) return PA_OK;
    float* base = static_workspace_address();
    if (!base) return PA_ERR_LAUNCH;
    pa_decode_args a = *args;
    a.mode = PA_MODE_V2;
    a.tmp_out = base;
    a.exp_sums = base + tmp;
    a.max_logits = base + tmp + stats;
    return pa_decode(&a, stream);
}
