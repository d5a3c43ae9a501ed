// pdl.cuh -- programmatic dependent launch between the library's kernels.
//
// A kernel launched with programmatic stream serialization may start while
// the kernel before it on the stream is still running: its CTAs set up
// (barriers, TMEM, tensor-map prefetch) and then wait in grid_dep_wait()
// until that kernel has completed and its memory is visible, before they
// touch any global memory it may have written or still reads.  A kernel
// lets the next one launch early by grid_dep_launch(), which the library's
// kernels call only after their own grid_dep_wait(): so what the kernels
// before the one ahead wrote is complete and visible from the start, and a
// dependent may read it before its wait.  Without grid_dep_launch() the
// next kernel starts when this one ends, as on an ordinary stream.
#pragma once

namespace mla {

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace mla
