"""Oracle package. TEST INFRASTRUCTURE ONLY.

A plain float64 CPU restatement of the TSP layer forward, written from the page
"Folding Tensor and Sequence Parallelism for Memory-Efficient Transformer
Training & Inference". Only the tests, the package smoke check and the
benchmark's CPU-baseline / reference legs may import it; the library never does.
"""
from .tsp_oracle import *  # noqa: F401,F403
from .tsp_oracle import __all__  # noqa: F401
