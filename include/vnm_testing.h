/*
 * Test support for libvnm: entry points that only tests call. The paper has
 * no counterpart; they exercise this library's own failure handling.
 */
#ifndef VNM_TESTING_H
#define VNM_TESTING_H

#include "vnm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * vnm_spmm on the tensor-core path, except that the first CTA never issues
 * the TMA loads of its pipeline stage number `skip_stage` (counted over the
 * tiles it takes). The waits on that stage are bounded (about 1 s): they run
 * out, every role of that CTA winds down, copies and MMAs already issued are
 * drained, TMEM is freed and VNM_ERR_TIMEOUT is recorded in the matrix's
 * status word (read it with vnm_get_status). C is then unspecified; the
 * device stays usable. Arguments as in vnm_spmm.
 * Errors: as vnm_spmm, plus VNM_ERR_UNSUPPORTED when the plan for this
 * product is not the tensor-core path or skip_stage < 0.
 */
vnm_status vnm_testing_spmm_skip_stage(vnm_matrix A, const void* B, int64_t ld_b, int64_t N, void* C,
                                       int64_t ld_c, vnm_dtype c_type, void* workspace, size_t workspace_bytes,
                                       int32_t skip_stage, vnm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VNM_TESTING_H */
