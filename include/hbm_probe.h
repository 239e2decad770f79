/*
 * hbm_probe.h -- C ABI of the HBM bandwidth probe (libhbmprobe.so).
 *
 * No counterpart in the paper: a measurement tool beside the optimizer.  It
 * times streaming kernels over caller-owned device buffers larger than L2 and
 * reports the bandwidth that each traffic mix reaches on this GPU -- the
 * ceiling the optimizer's bandwidth-bound kernels are set against:
 *   HBM_PROBE_COPY      read n 16-byte vectors, write them back elsewhere (1:1);
 *   HBM_PROBE_WRITE     write n 16-byte vectors;
 *   HBM_PROBE_READ      read n 16-byte vectors (one word per CTA written);
 *   HBM_PROBE_STEP_MIX  the fused optimizer step's mix: per 4 elements read
 *                       16 + 8 + 16 + 16 + 16 bytes from five buffers and write
 *                       16 + 16 + 16 + 8 bytes to four (18 : 14 bytes per element);
 *   HBM_PROBE_FIRST_MIX the first accumulate pass's: per 4 elements read 8 bytes,
 *                       write 16 (2 : 4 bytes per element);
 *   HBM_PROBE_ACC_MIX   a later accumulate pass's: per 4 elements read 16 + 8
 *                       bytes, write 16 (6 : 4 bytes per element);
 *   HBM_PROBE_BULK_STEP_MIX  the fused step's mix moved by bulk asynchronous
 *                       copies through shared memory, as the pipelined step
 *                       moves it (512-quad tiles, five stages, one copy
 *                       thread and eight compute warps per SM, 2,048 quads
 *                       per claim);
 *   HBM_PROBE_BULK_ACC_MIX   a later accumulate pass's mix the same way
 *                       (2,048-quad tiles, four stages, one tile per claim).
 * The first six kinds use 16-byte vector loads and stores.  Every kernel
 * takes its work from a counter the way the optimizer's passes do; the
 * counter returns to zero by itself at the end of each launch (the CTA
 * holding the last claim past the end resets it).  The bulk kinds bound every
 * wait on a shared-memory barrier (2 s); a wait that gives up makes the run
 * return -5.
 *
 * Buffers (device memory of the current device, 16-byte aligned, not
 * overlapping; the caller allocates them):
 *   COPY:     buf[0] source, buf[1] destination, each n x 16 bytes;
 *   WRITE:    buf[0], n x 16 bytes;
 *   READ:     buf[0], n x 16 bytes; buf[1] >= 4 bytes per CTA of the launch
 *             (hbm_probe_sink_bytes gives the size);
 *   STEP_MIX, BULK_STEP_MIX: n counts 4-element quads: buf[0] accumulator
 *             (16 B per quad), buf[1] gradient (8), buf[2..4] master, m, v (16
 *             each), buf[5] bf16 parameters (8);
 *   FIRST_MIX: n quads: buf[0] gradient (8 B per quad), buf[1] accumulator (16);
 *   ACC_MIX, BULK_ACC_MIX: n quads: buf[0] gradient (8 B per quad), buf[1]
 *             accumulator (16, read and written).
 * n must be a multiple of 4096 (64 KiB chunks of 16-byte vectors).
 *
 * hbm_probe_run times `reps` launches after `warmup` untimed ones with CUDA
 * events on `stream` and stores the mean milliseconds per launch in *ms and
 * the bytes one launch moves in *bytes.  It synchronises `stream`.  The
 * library's own scratch (the counter) is allocated on first use per device
 * and kept until exit.  Errors (negative): -1 invalid argument (NULL
 * pointers, unknown kind, n not a multiple of 4096, misaligned buffer),
 * -5 CUDA error; 0 on success.
 */
#ifndef HBM_PROBE_H
#define HBM_PROBE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HBM_PROBE_COPY 0
#define HBM_PROBE_WRITE 1
#define HBM_PROBE_READ 2
#define HBM_PROBE_STEP_MIX 3
#define HBM_PROBE_FIRST_MIX 4
#define HBM_PROBE_ACC_MIX 5
#define HBM_PROBE_BULK_STEP_MIX 6
#define HBM_PROBE_BULK_ACC_MIX 7

int hbm_probe_run(int kind, void *const *buf, uint64_t n, int warmup, int reps, void *stream, float *ms,
                  double *bytes);

/* Bytes buf[1] of HBM_PROBE_READ needs on the current device. */
int hbm_probe_sink_bytes(uint64_t *bytes);

#ifdef __cplusplus
}
#endif
#endif /* HBM_PROBE_H */
