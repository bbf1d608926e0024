"""CPU oracle for the FP4 paged-MQA indexer prefill (test infrastructure only).

Only tests/, the smoke check and the benchmark's CPU-baseline leg import this
package.  The product path never does, and this package imports nothing from
the product.
"""
from .oracle import (build, e2m1_value, ue8m0_value, row_logits, row_scores, select,
                     prefill_rows, threads, OracleError)

__all__ = ["build", "e2m1_value", "ue8m0_value", "row_logits", "row_scores", "select",
           "prefill_rows", "threads", "OracleError"]
