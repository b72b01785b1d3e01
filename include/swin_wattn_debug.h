/*
 * swin_wattn fault-injection build: one extra entry point, exported only by
 * libswin_wattn_debug.so (the library compiled with SWIN_WATTN_FAULT_INJECTION). The
 * default library libswin_wattn.so neither exports it nor contains the injection code.
 *
 * The pages have no counterpart: this exists to test the library's failure handling.
 * Every device-side wait of the library's kernels (on an mbarrier that a copy, a tensor-
 * core commit or another warp completes) is bounded; when one runs out, the kernel stops
 * its own work, lets its copies and tensor-core operations in flight complete (with the
 * same bound), releases its tensor memory, sets an error word and returns, so the CUDA
 * context stays usable. The error reaches the caller as SWIN_WATTN_ERR_TIMEOUT from
 * swin_wattn_device_status (attention kernels) or as bit 0 of the status word of the
 * GEMM steps.
 */
#ifndef SWIN_WATTN_DEBUG_H
#define SWIN_WATTN_DEBUG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum swin_wattn_fault_site {
  SWIN_WATTN_FAULT_NONE = 0,
  /* mma.sync forward with copy-engine tiles (7x7 windows, bf16): in every CTA, on the first
     window it gathers by cp.async (a window of the last window column of a shifted layer),
     thread 0 does not arrive on that window's stage barrier. */
  SWIN_WATTN_FAULT_FWD_MMA_SYNC = 1,
  /* tcgen05 forwards: row warp 0 does not arrive on the "P written" barrier of the first
     pair of windows (7x7) or of the first window (12x12), so the MMA warp's wait runs out,
     then the other roles' waits. */
  SWIN_WATTN_FAULT_FWD_TCGEN05 = 2,
  /* GEMM steps (qkv projection, output projection): the MMA thread does not commit the
     "accumulator full" barrier of its first output tile, so the epilogue warps' wait runs
     out, then the other roles' waits. */
  SWIN_WATTN_FAULT_GEMM = 3
};

/*
 * Arm `site` (SWIN_WATTN_FAULT_*; NONE disarms) for every later launch of that kernel,
 * process-wide, and set the bound of every device-side wait to `wait_limit_ns`
 * (1e3 .. 1e10; the default library's bound is 1e9). Host-side only; call it between
 * launches. Returns SWIN_WATTN_OK or SWIN_WATTN_ERR_INVALID_ARG.
 */
int swin_wattn_debug_set_fault(int site, int64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* SWIN_WATTN_DEBUG_H */
