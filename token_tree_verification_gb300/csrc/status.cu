// Names of the library's status codes.
#include "../../include/spec_tree.h"

extern "C" const char *spec_status_string(int code) {
  switch (code) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_NULL: return "SPEC_ERR_NULL: a required pointer is NULL";
    case SPEC_ERR_SHAPE: return "SPEC_ERR_SHAPE: a size argument is out of range or unsupported";
    case SPEC_ERR_DTYPE: return "SPEC_ERR_DTYPE: unknown dtype";
    case SPEC_ERR_TREE_TOO_LARGE: return "SPEC_ERR_TREE_TOO_LARGE: bad tree size or offsets";
    case SPEC_ERR_BAD_PARENT: return "SPEC_ERR_BAD_PARENT: malformed parent array";
    case SPEC_ERR_TOKEN_RANGE: return "SPEC_ERR_TOKEN_RANGE: token outside [0, V)";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE: workspace missing or too small";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA: CUDA call or launch failed";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT: a bounded device wait ran out";
    case SPEC_ERR_PREFIX_RANGE: return "SPEC_ERR_PREFIX_RANGE: prefix does not fit the cache";
    case SPEC_ERR_ALIGNMENT: return "SPEC_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case SPEC_ERR_INDEX: return "SPEC_ERR_INDEX: a computed index fell outside its buffer";
    default: return "unknown spec_status";
  }
}

extern "C" int spec_build_checked(void) {
#ifdef SPEC_CHECKED
  return 1;
#else
  return 0;
#endif
}
