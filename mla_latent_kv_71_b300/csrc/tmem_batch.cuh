// tmem_batch.cuh -- TMEM loads issued back to back with one wait.
//
// tmem_ld32 (ptx.cuh) waits for its own load inside the same statement; a
// thread that needs several column blocks pays one TMEM round trip per
// block.  These issue the loads without waiting, so that several are in
// flight, then wait once; tmem_reg_fence makes the compiler treat the
// destination registers as written at that point, so no use of them is
// scheduled before the wait.
#pragma once

#include <cstdint>

namespace mla {

// TMEM -> registers, 32 lanes x 32 columns, without the wait (issue several,
// then tmem_wait_ld and tmem_reg_fence on the registers before their use).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Keeps every use of r after the wait: the compiler sees r rewritten here.
__device__ __forceinline__ void tmem_reg_fence(uint32_t* r, int n) {
#pragma unroll
    for (int i = 0; i < n; ++i) asm volatile("" : "+r"(r[i]));
}

}  // namespace mla
