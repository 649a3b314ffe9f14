/*
 * qsa_selftest.h -- failure-detection self-test of libqsa (not part of the
 * hot path; declared apart from qsa.h so that no decode caller reaches it).
 *
 * The notes ask the checkpoint to show both a clean completion and a
 * non-completion gate ([AFN-017] Retrieval capsule: "non-completion, and
 * clean-completion gates").  On the GPU a non-completion is a copy that never
 * lands: every wait of the scorer on its copy ring is bounded in time, and
 * a wait that runs out sets QSA_DEVERR_WAIT_TIMEOUT in the workspace's error
 * word instead of trapping or hanging.  This call makes that happen on
 * purpose, without a fault: it runs the raw-key scorer with its copy
 * producer switched off, so nothing is ever issued and the first wait of
 * every CTA runs out after wait_ns.
 */
#ifndef QSA_SELFTEST_H
#define QSA_SELFTEST_H

#include "qsa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Arguments as qsa_score_groups (which reads in->q_idx, idx_keys,
 * key_offset, visible), plus wait_ns: the limit of each copy wait, in
 * nanoseconds of wall time (1 ..= 1e9).  The launch issues no copy; each
 * CTA's first wait runs out, the CTA sets QSA_DEVERR_WAIT_TIMEOUT, has
 * nothing in flight to wait for, writes no score and exits.  The call takes
 * about wait_ns on the GPU.  Afterwards the context and the workspace stay
 * usable: qsa_check_errors reports the flag and clears it.  The per-SM
 * scorer weights of the workspace are neither read nor changed.
 * Returns QSA_ERR_INVALID_ARG for wait_ns outside 1 ..= 1e9. */
qsa_status qsa_selftest_copy_timeout(const qsa_dims *dims, const qsa_inputs *in, float *scores, void *ws,
                                     size_t ws_bytes, uint64_t wait_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_SELFTEST_H */
