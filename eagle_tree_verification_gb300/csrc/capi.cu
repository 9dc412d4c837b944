// Library-wide entry points of the C ABI (status strings, version).
#include "common.cuh"

extern "C" const char* eagle_status_string(int status) {
  switch (status) {
    case EAGLE_OK: return "ok";
    case EAGLE_ERR_INVALID_ARG: return "invalid argument";
    case EAGLE_ERR_INVALID_TREE: return "invalid tree";
    case EAGLE_ERR_UNSUPPORTED: return "unsupported shape";
    case EAGLE_ERR_NUMERIC: return "numeric error";
    case EAGLE_ERR_TIMEOUT: return "device wait timed out";
    case EAGLE_ERR_CUDA: return "CUDA error";
    case EAGLE_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

extern "C" const char* eagle_version(void) { return "eagle-tree-verify-gb300 0.1 (sm_103a)"; }
