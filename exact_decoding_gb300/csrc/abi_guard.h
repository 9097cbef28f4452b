// No C++ exception may leave an entry point of the C ABI.  Each exported
// function runs its body through abi_guard.  A std::bad_alloc (a host
// container or string that could not grow) becomes LA_ERR_OOM.  Any other
// exception (for example std::system_error from a mutex) becomes
// LA_ERR_STATE.  Both set the thread's last-error message when that is
// still possible.
#pragma once

#include <cstdio>
#include <exception>
#include <new>

#include "../../include/la.h"

namespace la {

int set_last_error(int code, const char *msg);

template <typename Body>
int abi_guard(const char *where, Body &&body) noexcept {
    int code = LA_ERR_STATE;
    const char *what = "unexpected C++ exception";
    try {
        return body();
    } catch (const std::bad_alloc &) {
        code = LA_ERR_OOM;
        what = "host allocation failed";
    } catch (...) {
    }
    try {
        char msg[160];
        std::snprintf(msg, sizeof(msg), "%s: %s", where, what);
        set_last_error(code, msg);
    } catch (...) {
    }
    return code;
}

}  // namespace la
