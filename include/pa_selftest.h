/*
 * pa_selftest.h -- test hooks of the paged-attention library (not part of the attention API).
 *
 * Every wait inside the library's kernels is bounded: when the expected arrival never comes,
 * the waiting thread gives up after a limit, sets the timeout bit of the device error word and
 * returns, so a lost copy or a broken protocol never hangs the GPU (pa.h, pa_set_wait_limit).
 * The hook below lets a test drive that path to its end on purpose, without a fault and without
 * any copy in flight, and then check that the status comes back and the context stays usable.
 */
#ifndef PA_SELFTEST_H_
#define PA_SELFTEST_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pa_selftest_wait_timeout -- launch, on `stream` (a cudaStream_t), one warp whose lane 0
 * initialises an mbarrier that nothing ever arrives on and waits on its first phase with the
 * library's bounded wait and the given limit.  The wait runs out after limit_ns, sets the
 * timeout bit (1) of the device error word and the kernel returns; no memory copy is ever
 * issued.  pa_get_device_error then returns PA_ERR_TIMEOUT.  limit_ns must be in
 * [PA_WAIT_LIMIT_MIN_NS, 100 ms] (else PA_ERR_INVALID_ARG, nothing launched).  Asynchronous.
 */
int pa_selftest_wait_timeout(uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_SELFTEST_H_ */
