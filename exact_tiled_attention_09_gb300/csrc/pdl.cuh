// Programmatic dependent launch between the kernels of one call.
//
// A kernel launched with programmatic stream serialization is launched as
// the kernel before it on the stream drains (its launch overlaps that
// kernel's last blocks).  Before it touches anything that kernel writes it
// executes griddepcontrol.wait, which returns once the earlier grid has
// completed and its memory operations are visible.  No kernel here triggers
// its dependants early (griddepcontrol.launch_dependents): measured, a
// dependant resident early takes registers or threads that the running
// grid's blocks need.  In a kernel launched without the attribute the wait
// does nothing.
#pragma once

#include <cuda_runtime.h>

namespace fa {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace fa
