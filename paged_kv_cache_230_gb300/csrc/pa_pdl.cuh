// Programmatic dependent launch between kernels of one stream: a kernel
// launched with the programmatic-serialization attribute may start while the
// kernel before it runs, once every CTA of that kernel has signalled
// (pdl_trigger) or exited; its threads that read what the earlier kernel
// writes wait for that kernel's completion and memory first (pdl_wait).
// Launched without the attribute, the wait returns at once.
#pragma once

namespace pa {

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace pa
