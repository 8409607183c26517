"""Seeded synthetic input generation shared by the tests, the bench and the oracle checks.

`workloads` draws the request structure and small inputs; `ih12.h` defines the
counter-based generator of the bulk tensors, compiled for the host
(`gen_host.c`, via gcc) and for the GPU (`gen_dev.cu`, via nvcc).  This
package holds none of the routing method's arithmetic.
"""
from .workloads import (Batch, Workload, make_workload, make_custom, make_calibration,  # noqa: F401
                        CONFIGS, calib_signatures, kmeans_seed_rows)
from .native import (build, host_logits, host_logit_rows, host_hidden, host_wgate,  # noqa: F401
                     dev_logits, dev_hidden, dev_wgate)
