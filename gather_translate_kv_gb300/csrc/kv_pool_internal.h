// The pool handle behind kv_pool_t, shared by the translation units that
// implement the C ABI. Not part of the public interface.
#pragma once

#include <stdint.h>

#include "kv_common.cuh"
#include "kv_layout.h"
#include "kv_pool.h"

struct kv_pool {
  kv_pool_desc desc;
  gtkv::Layout lay;
  uint8_t* raw;
  int64_t raw_bytes;
  int owns_raw;
  int32_t* d_err;
  int device;
  int sm_count;
  gtkv::DevPool dev;
};
