// status.cuh -- the device status word shared by every kernel of the library.
//
// Kernels never trap, assert or spin forever.  A bounded wait that gives up,
// or an out-of-range page id / sequence length found on the device, raises
// the status word (first error wins) and the kernel winds down.  While the
// word is raised, later kernels of this library on the same device return
// early; mla_get_device_status() reads and clears it.
#pragma once

#include <cstdint>

namespace mla {

// Device-side error kinds (low 8 bits of the word); bits 8..31 hold a detail.
enum : uint32_t {
    MLA_DEV_OK = 0,
    MLA_DEV_TIMEOUT = 1,
    MLA_DEV_BOUNDS = 2,
};

// A bounded wait gives up after this much wall time (globaltimer, ns) by
// default.  The limit in use is g_wait_limit_ns, which the host may shorten
// (mla_set_wait_limit) to exercise the failure path; teardown waits for
// copies already in flight keep their own fixed limits.
constexpr uint64_t MLA_WAIT_LIMIT_NS = 2000000000ull;

// Defined once: the library is a single translation unit (mla_lib.cu).
__device__ uint32_t g_device_status = 0u;
// In constant memory: every wait reads it, and a constant-cache read costs
// next to nothing (the host changes it only between calls).
__constant__ uint64_t g_wait_limit_ns = MLA_WAIT_LIMIT_NS;

__device__ __forceinline__ uint64_t wait_limit_ns() { return g_wait_limit_ns; }

__device__ __forceinline__ bool device_status_raised() {
    return *reinterpret_cast<volatile uint32_t*>(&g_device_status) != 0u;
}

__device__ __forceinline__ void raise_device_status(uint32_t kind, uint32_t detail) {
    atomicCAS(&g_device_status, 0u, (kind & 0xFFu) | (detail << 8));
}

// The debug build (MLA_CHECKS=1, libmla_checks.so) checks each kernel's work
// split against the shapes: a violated condition raises MLA_DEV_BOUNDS with
// the given detail (0x7x).  Release builds compile the checks away.
#ifndef MLA_CHECKS
#define MLA_CHECKS 0
#endif

__device__ __forceinline__ void check_split(bool ok, uint32_t detail) {
#if MLA_CHECKS
    if (!ok) raise_device_status(MLA_DEV_BOUNDS, detail);
#else
    (void)ok;
    (void)detail;
#endif
}

// Debug build: fill `bytes` (a multiple of 16) of shared memory at p with
// all-ones bytes (NaN as fp32 and bf16) from every thread of the block, then
// order those writes before any later TMA copy into the same bytes; a read
// of shared memory that no copy wrote then shows up as NaN in the results.
// The caller synchronises the block afterwards.
__device__ __forceinline__ void poison_smem(void* p, uint32_t bytes) {
#if MLA_CHECKS
    uint4* q = static_cast<uint4*>(p);
    for (uint32_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) q[i] = make_uint4(~0u, ~0u, ~0u, ~0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#else
    (void)p;
    (void)bytes;
#endif
}

}  // namespace mla
