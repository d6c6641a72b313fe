// diag.h -- MLQ_DIAG=1: one line on stderr per distinct (entry point, shape,
// kernel, launch geometry), so that a caller can see which of the several
// kernels behind an entry point ran and how it was laid out.  Off by
// default; when off every call below returns at once.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace mlq {

bool diag_on();
// Called by a C-ABI entry point: its name and the shape it was given.
void diag_entry(const char *entry, const char *fmt, ...);
// Called by a launcher before it launches: the route or geometry it chose
// (stages, chunks, rows per CTA ...), appended to the next launch line.
void diag_note(const char *fmt, ...);
// Called at every kernel launch: prints the line once per distinct text.
void diag_launch(const void *kern, dim3 grid, dim3 block, size_t smem, int cluster, bool pdl);
// The same for a cudaLaunchKernelEx configuration (cluster and dependent-
// launch attributes read from it).
inline void diag_launch_cfg(const void *kern, const cudaLaunchConfig_t &cfg) {
  if (!diag_on()) return;
  int cluster = 1;
  bool pdl = false;
  for (unsigned i = 0; i < cfg.numAttrs; ++i) {
    if (cfg.attrs[i].id == cudaLaunchAttributeClusterDimension)
      cluster = static_cast<int>(cfg.attrs[i].val.clusterDim.x * cfg.attrs[i].val.clusterDim.y *
                                 cfg.attrs[i].val.clusterDim.z);
    if (cfg.attrs[i].id == cudaLaunchAttributeProgrammaticStreamSerialization)
      pdl = cfg.attrs[i].val.programmaticStreamSerializationAllowed != 0;
  }
  diag_launch(kern, cfg.gridDim, cfg.blockDim, cfg.dynamicSmemBytes, cluster, pdl);
}

}  // namespace mlq
