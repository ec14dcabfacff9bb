// Decode with library-static scratch: the allocation-free variant of the
// split-KV decode (see attn_decode_noalloc in include/attn.h).
//
// The split-KV decode needs scratch for its per-chunk partial results.  The
// regular entry point keeps that scratch in a buffer it allocates on first
// use; this variant uses a fixed array compiled into the library instead, so
// a call never allocates or frees device memory.  The array is a file-scope
// __device__ variable: every GPU that loads this part of the library holds it
// until the process exits.
#include "kernels.h"

#include <cuda_runtime.h>

#include <mutex>

// Scratch for the decode partials: B*H*splits*(D + 2) floats must fit.
static __device__ __align__(256) unsigned char g_decode_scratch[attn::kDecodeNoAllocScratchBytes];

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];

}  // namespace

// Device address of the scratch array on the current device.  In host code
// the array's name only stands in for the symbol, so the address is looked up
// once per device (with that device current) and cached.
cudaError_t decode_noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

// The regular decode kernels (bf16, or fp32 when f32), with their partials in
// the static scratch.  The partials need no clearing: every chunk the combine
// step reads is written by the same call first.
cudaError_t launch_decode_noalloc(DecodeArgs a, bool f32) {
    void *scratch = nullptr;
    cudaError_t e = decode_noalloc_scratch(&scratch);
    if (e != cudaSuccess) return e;
    const size_t o_bytes = static_cast<size_t>(a.B) * a.H * a.n_split * a.D * sizeof(float);
    a.part_o = static_cast<float *>(scratch);
    a.part_ml = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + o_bytes);
    return f32 ? launch_decode_f32(a) : launch_decode(a);
}

}  // namespace attn
