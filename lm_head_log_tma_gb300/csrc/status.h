// Status codes shared by host and device code of the library.  The public
// copies of these values live in include/rlloss.h; this header only pulls
// them in for the CUDA sources.
#pragma once
#include "../../include/rlloss.h"
