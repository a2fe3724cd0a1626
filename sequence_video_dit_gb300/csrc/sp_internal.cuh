// Internal helpers shared by the library's translation units.
#pragma once

#include <stddef.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "sp_api.h"

namespace sp {

// Workspace header layout (SP_WORKSPACE_HEADER_BYTES = 256 bytes, ints).
struct WorkspaceHeader {
    int status;                      // sticky device status (first error wins)
    int ticket;                      // CTAs of the running exchange that have finished
    int counters[SP_MAX_RANKS];      // per-destination completion counters ("barrier")
    int observed[SP_MAX_RANKS];      // counters seen by the last CTA of the last exchange
    int launches;                    // completed exchange launches
    int grid;                        // CTAs of the last exchange launch
    int kv_stall;                    // test hook, SP_WORKSPACE_KV_STALL_OFFSET: > 0 stops the
                                     // attention's K/V loads after kv_stall - 1 of them
    int reserved[64 - 5 - 2 * SP_MAX_RANKS];
};
static_assert(sizeof(WorkspaceHeader) == SP_WORKSPACE_HEADER_BYTES, "header size");
static_assert(offsetof(WorkspaceHeader, kv_stall) == SP_WORKSPACE_KV_STALL_OFFSET, "stall word offset");

// Thread-local error message; returns `code` for chaining.
int set_error(int code, const char *fmt, ...);
inline int ok() { return SP_OK; }

// Device properties of the current device (cached per device).
struct DeviceInfo {
    int device;
    int num_sms;
    int cc_major, cc_minor;
    size_t l2_bytes;
    size_t max_smem_optin;
};
int device_info(DeviceInfo *out);

#define SP_CUDA_CHECK(expr)                                                                  \
    do {                                                                                     \
        cudaError_t _e = (expr);                                                             \
        if (_e != cudaSuccess)                                                               \
            return ::sp::set_error(SP_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(_e)); \
    } while (0)

// Kernels launched by this library (sp_launch_count()).
void count_launch();

// After a launch: count it and report launch-configuration errors without
// synchronising.
inline int check_launch(const char *what) {
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(SP_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
    return SP_OK;
}

// Largest power-of-two vector width (<= 16 bytes) dividing every value.
inline int vector_width(uint64_t a) {
    int v = 16;
    while (v > 1 && (a % (uint64_t)v) != 0) v >>= 1;
    return v;
}

__device__ __forceinline__ void set_device_status(int *status, int code) {
    atomicCAS(status, 0, code);
}

}  // namespace sp
