// Library-internal: the thread-local last-error text returned by mosaic_last_error_string().
#pragma once

namespace mosaic {
void set_last_error(const char* msg);
}  // namespace mosaic
