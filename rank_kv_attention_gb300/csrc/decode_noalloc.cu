// lrkv_decode_noalloc: lrkv_decode for callers that cannot allocate device
// memory.  The decode's scratch (launch plan, private queries and per-segment
// partial softmax states) lives in one file-scope device array that is part
// of the library image, so the caller passes only inputs and outputs.
#include "decode_kernels.cuh"

namespace lrkv {

// Device-resident scratch shared by every lrkv_decode_noalloc call on a GPU.
// In host code `g_noalloc_scratch` names a host-side stand-in, not a device
// address: its device address is obtained with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LRKV_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up on
// every call with that device current.  The first lookup on a device loads
// the library's device code there (CUDA loads modules lazily), which is when
// the array's memory is committed; later lookups are a table read.  Looking
// it up each time, instead of caching it, keeps the address right after the
// device's primary context has been reset and the module loaded again.
// Returns nullptr (and sets *err) on failure.
void *noalloc_scratch_address(cudaError_t *err) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) {
        cudaGetLastError();  // reset the last-error state so later CUDA calls start clean
        return nullptr;
    }
    return p;
}

}  // namespace lrkv
