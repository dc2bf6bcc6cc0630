// Error reporting, version and device-error query of the libqw C ABI.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <string>

#include "common.cuh"

namespace qw {

static thread_local std::string g_last_error;

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return QW_OK;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("QW_NO_PDL");
    return !(v && v[0] == '1');
  }();
  return on;
}

// defined next to the kernels that own a bounded-wait error word
unsigned int take_tc_timeouts();
unsigned int take_attn_timeouts();
unsigned int take_prefill_timeouts();
unsigned int take_dstep_errors();

}  // namespace qw

extern "C" int qw_abi_version(void) { return 9; }

extern "C" const char* qw_last_error_string(void) { return qw::g_last_error.c_str(); }

extern "C" int qw_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return qw::set_error(QW_ERR_CUDA, "qw_device_error: %s", cudaGetErrorString(e));
  const unsigned int gemm = qw::take_tc_timeouts(), dec_word = qw::take_attn_timeouts(),
                     pre = qw::take_prefill_timeouts(), step = qw::take_dstep_errors();
  const unsigned int dec = dec_word & ~qw::kErrContextOverflow;
  if (gemm | dec | pre | step)
    return qw::set_error(QW_ERR_TIMEOUT,
                         "a bounded device-side wait timed out (gemm 0x%x, decode attention 0x%x, prefill attention "
                         "0x%x, decode step 0x%x)",
                         gemm, dec, pre, step);
  if (dec_word & qw::kErrContextOverflow)
    return qw::set_error(QW_ERR_INVALID_ARG,
                         "decode attention: a context_lens entry exceeded the call's max_context; the keys past it "
                         "were not read");
  return QW_OK;
}
