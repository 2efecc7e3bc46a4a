/*
 * msa_profile.h -- per-kernel timing of the MSA library (tracing aid) and a
 * test hook for its timeout path.
 *
 * Between msa_profile_begin() and msa_profile_end() every kernel launched by
 * an msa_* entry point is bracketed by a pair of CUDA events recorded on the
 * stream it is launched on. msa_profile_end() waits for those events and
 * returns, per kernel name, the launch count and the summed device time.
 * Host-side bookkeeping only; no extra device work is enqueued. Not
 * thread-safe against concurrent begin/end calls from several threads.
 */
#ifndef MSA_PROFILE_H_
#define MSA_PROFILE_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  const char* name; /* static kernel name */
  int launches;
  double total_ms;
} msa_kernel_time_t;

/* Starts recording (drops earlier records). Returns 0. */
int msa_profile_begin(void);

/* Stops recording, synchronises the recorded events and writes up to
 * `max_entries` per-kernel totals to `out` (in first-launch order). Returns
 * the number of distinct kernels, or -1 if an event query failed. */
int msa_profile_end(msa_kernel_time_t* out, int max_entries);

/* Test hook for the bounded-wait timeout path (no counterpart in the paper).
 * While enabled (enable != 0), every launch of the prefill attention kernel
 * (tensor-core path) and of the decode attention kernel first waits on a
 * device barrier that nothing completes. That wait gives up after about a
 * millisecond; the kernel then records MSA_ERR_TIMEOUT in the workspace status,
 * lets the copies and matrix products it has in flight finish, frees its
 * tensor memory and returns. The outputs of such a call are unspecified; the
 * workspace stays usable for the next call once msa_read_status() has cleared
 * the status. Process-wide, for all devices and threads; returns the previous
 * setting. Off by default. */
int msa_debug_inject_timeout(int enable);

#ifdef __cplusplus
}
#endif

#endif /* MSA_PROFILE_H_ */
