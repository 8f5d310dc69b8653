// api.cu -- status strings and version of the C ABI declared in fp8q.h.
#include "fp8q.h"

extern "C" const char *fp8q_status_string(fp8q_status s) {
  switch (s) {
    case FP8Q_OK: return "ok";
    case FP8Q_ERR_INVALID: return "invalid argument (null pointer or unknown enum value)";
    case FP8Q_ERR_SHAPE: return "invalid shape (negative size, K/T not a multiple of 128, "
                                "leading dimension too small, or size limit exceeded)";
    case FP8Q_ERR_ALIGN: return "misaligned pointer or leading dimension (16-byte rules)";
    case FP8Q_ERR_UNSUPPORTED: return "unsupported device (needs sm_103 with enough shared memory)";
    case FP8Q_ERR_CUDA: return "CUDA runtime error";
    case FP8Q_ERR_TIMEOUT: return "a device-side wait timed out";
  }
  return "unknown status";
}

extern "C" int fp8q_version(void) { return 100; }
