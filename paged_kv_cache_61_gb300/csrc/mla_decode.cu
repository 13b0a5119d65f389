// Absorbed-MLA paged decode for sm_103a (tcgen05 / TMEM). Not built yet: every
// MLA problem is reported as unsupported.
#include <cuda_runtime.h>

#include "pda_internal.h"

namespace pda {

bool mla_supported(const pda_problem&, std::string* why) {
  *why = "MLA decode is not available in this build";
  return false;
}

int mla_ctas_per_sm(const pda_problem&) { return 1; }
int mla_heads_per_cta(const pda_problem& p) { return p.num_q_heads; }

int launch_mla_decode(const Plan&, const MlaArgs&, const Workspace&, void*) {
  return cudaErrorNotSupported;
}

}  // namespace pda
