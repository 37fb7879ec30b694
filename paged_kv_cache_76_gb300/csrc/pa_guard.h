// Host-side guard for the C entry points that allocate host memory (the
// block allocator, the VMM bookkeeping): a failed allocation must not leave
// a C call as an exception (that ends the process), it becomes a status.
#pragma once

#include <new>

#include "pa.h"

template <class F>
inline int pa_guarded(F&& body) noexcept {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    return PA_ERR_HOST_MEMORY;
  } catch (...) {
    return PA_ERR_INVALID;
  }
}
