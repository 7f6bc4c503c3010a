// Test helper: a kernel that lets its programmatic dependents start at once and writes new sequence
// lengths only ~delay_ns later, so that a decode launched right after it (a programmatic dependent)
// computes its split from the old lengths before its dependency wait.  The delay is a bounded spin
// on the global timer.
#include <cuda_runtime.h>

#include <cstdint>

__global__ void write_lengths_late(int* lens, const int* new_lens, int n, unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;");
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < delay_ns);
  for (int i = threadIdx.x; i < n; i += blockDim.x) lens[i] = new_lens[i];
}

extern "C" int launch_write_lengths_late(int* lens, const int* new_lens, int n, unsigned long long delay_ns,
                                         void* stream) {
  write_lengths_late<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(lens, new_lens, n, delay_ns);
  return static_cast<int>(cudaGetLastError());
}
