// fa_get_device_status: the short form of fa_check_device_status (include/fa.h).
#include "fa.h"

fa_status fa_get_device_status(fa_stream_t stream) { return fa_check_device_status(stream, nullptr); }
