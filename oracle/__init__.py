"""Float64 CPU oracle for the batched block-preconditioner step of DASH-style Shampoo.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
restatement of what the GPU library computes.  Only the test-suite, the smoke
check in ``__graft_entry__.smoke`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import it.  The product path (the CUDA library and its Python
binding) never imports, links or executes anything under ``oracle/``, and this
package imports nothing from the product path: the two share no code.

Sources.  The method is described by five web pages about the paper
"DASH: Faster Shampoo via Batched Block Preconditioning and Efficient
Inverse-Root Solvers" (arXiv 2602.02016).  They are cited by title and section:

  [pt]  gist.science/pt, "Resumo Tecnico: DASH - Shampoo Mais Rapido via
        Pre-condicionamento de Blocos em Lote ..."  (sections "Definicao do
        Problema", "Metodologia" 1 and 2, "Principais Contribuicoes",
        "Resultados Experimentais")
  [fr]  gist.science/fr, same technical summary in French ("Methodologie")
  [ko]  gist.science/ko, same technical summary in Korean
  [tg]  tgviewer.app, Telegram channel quant_prune_distill, post 646
  [abs] arxivdaily.com, the authors' abstract

The pages name the solvers (Coupled Newton, Newton-Denman-Beavers,
Chebyshev/Clenshaw, multi-vector power iteration) and their properties but print
no update formulas.  Every recurrence here is the plainest textbook reading
consistent with those properties; each module states which reading it takes.

Parity pins.  Every function is pinned in ``tests/test_oracle_pins.py`` by
closed forms, invariants, library routines that compute the same quantity by a
different algorithm, or brute force on tiny inputs.  No function here is
"parity unpinned".
"""

from .shampoo64 import (accumulate, apply_preconditioner, frobenius_norm, pack_blocks,
                        power_lambda, unpack_blocks, update_weights)
from .roots64 import (
    evd_inv_root,
    cn_inv_root,
    ndb_inv_root,
    cheb_coeffs,
    cheb_inv_root,
)
from .select64 import (DEFAULT_TIERS, auto_inv_root, condition_estimate, lambda_min_estimate,
                       select_tiers)

__all__ = [
    "accumulate",
    "apply_preconditioner",
    "frobenius_norm",
    "power_lambda",
    "evd_inv_root",
    "cn_inv_root",
    "ndb_inv_root",
    "cheb_coeffs",
    "cheb_inv_root",
    "pack_blocks",
    "unpack_blocks",
    "update_weights",
    "DEFAULT_TIERS",
    "lambda_min_estimate",
    "condition_estimate",
    "select_tiers",
    "auto_inv_root",
]
