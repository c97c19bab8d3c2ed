"""Expert-major chunked MoE prefill layer for GB300 (sm_103a).

The layer lives in the C-ABI library libmoe_prefill.so (include/moe_prefill.h, sources in csrc/); `binding`
marshals arguments to it. `workloads` draws seeded synthetic inputs. Importing this package loads nothing; the
library is built (nvcc) and loaded on first use of `binding.lib()`.
"""

__all__ = ["binding", "build", "workloads"]
