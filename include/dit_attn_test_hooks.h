/*
 * dit_attn_test_hooks.h -- test-only entry point of libdit_attn_testhooks.so.
 *
 * That library is built from the same sources as libdit_attn.so (and exports the same
 * calls), with DIT_TEST_HOOKS defined for the attention kernels. It exists so that tests can
 * make a bounded wait run out without faulting or hanging the GPU, and check that the kernel
 * gives up cleanly: it records a status bit, lets its in-flight copies and MMAs land, frees
 * its tensor memory and returns. The product library libdit_attn.so contains none of this.
 * The pages have no counterpart; this is test infrastructure for the library's own
 * failure handling.
 */
#ifndef DIT_ATTN_TEST_HOOKS_H_
#define DIT_ATTN_TEST_HOOKS_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Sets, on the current device, the limit of every bounded wait in the attention kernels
 * (nanoseconds of %globaltimer; the product build uses 2 s) and the number of the load that
 * a kernel's K/V producer counts but never issues (-1 = none). In the attention kernel that
 * is a K/V ring load, numbered K_0, K_1, V_0, K_2, V_1, ... per CTA; in the short-KV
 * cross-attention kernel a fill (the keys and values of one head), numbered 0, 1, ... per
 * CTA. With skip_load = 0 the first S product's wait runs out after wait_limit_ns, and the
 * call ends with a timeout bit in the status word (dit_device_status of this library).
 * Synchronises the device.
 * Returns 0, -1 (wait_limit_ns == 0) or -4 (a CUDA call failed). */
int dit_test_set_wait_hooks(unsigned long long wait_limit_ns, int skip_load);

#ifdef __cplusplus
}
#endif

#endif /* DIT_ATTN_TEST_HOOKS_H_ */
